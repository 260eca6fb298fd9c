// Kernel instantiations for d_head = 64, no mask (2 to 4 K/V ring slots).
#include "fa_launch.h"

namespace fa {
FA_DEFINE_LAUNCH(64, 2, false, false)
FA_DEFINE_LAUNCH(64, 3, false, false)
FA_DEFINE_LAUNCH(64, 4, false, false)
FA_DEFINE_LAUNCH(64, 2, true, false)
FA_DEFINE_LAUNCH(64, 3, true, false)
FA_DEFINE_LAUNCH(64, 4, true, false)
}  // namespace fa
