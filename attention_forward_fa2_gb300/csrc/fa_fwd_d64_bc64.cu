// Kernel instantiations for d_head = 64 with a 64-key tile, no mask (two to
// four K/V ring slots of 16 KiB).
#include "fa_launch.h"

namespace fa {
FA_DEFINE_LAUNCH(64, 64, 2, false, false)
FA_DEFINE_LAUNCH(64, 64, 3, false, false)
FA_DEFINE_LAUNCH(64, 64, 4, false, false)
FA_DEFINE_LAUNCH(64, 64, 2, true, false)
FA_DEFINE_LAUNCH(64, 64, 3, true, false)
FA_DEFINE_LAUNCH(64, 64, 4, true, false)
}  // namespace fa
