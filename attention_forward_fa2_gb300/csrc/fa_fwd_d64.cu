// Kernel instantiations for d_head = 64 (2 to 4 K/V ring slots).
#include "fa_launch.h"

namespace fa {
FA_DEFINE_LAUNCH(64, 2, false)
FA_DEFINE_LAUNCH(64, 3, false)
FA_DEFINE_LAUNCH(64, 4, false)
FA_DEFINE_LAUNCH(64, 2, true)
FA_DEFINE_LAUNCH(64, 3, true)
FA_DEFINE_LAUNCH(64, 4, true)
}  // namespace fa
