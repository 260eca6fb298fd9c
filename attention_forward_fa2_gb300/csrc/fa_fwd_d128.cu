// Kernel instantiations for d_head = 128.
#include "fa_launch.h"

namespace fa {
FA_DEFINE_LAUNCH(128, 2, false)
FA_DEFINE_LAUNCH(128, 3, false)
FA_DEFINE_LAUNCH(128, 4, false)
FA_DEFINE_LAUNCH(128, 2, true)
FA_DEFINE_LAUNCH(128, 3, true)
FA_DEFINE_LAUNCH(128, 4, true)
}  // namespace fa
