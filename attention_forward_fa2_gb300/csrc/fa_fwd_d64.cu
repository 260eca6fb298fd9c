// Kernel instantiations for d_head = 64, no mask (key tile 128 or 64, two to
// four K/V ring slots).
#include "fa_launch.h"

namespace fa {
FA_DEFINE_LAUNCH(64, 128, 2, false, false)
FA_DEFINE_LAUNCH(64, 128, 3, false, false)
FA_DEFINE_LAUNCH(64, 128, 4, false, false)
FA_DEFINE_LAUNCH(64, 128, 2, true, false)
FA_DEFINE_LAUNCH(64, 128, 3, true, false)
FA_DEFINE_LAUNCH(64, 128, 4, true, false)
}  // namespace fa
