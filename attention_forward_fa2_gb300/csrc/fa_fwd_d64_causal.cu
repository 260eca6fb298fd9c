// Kernel instantiations for d_head = 64 with the causal mask.
#include "fa_launch.h"

namespace fa {
FA_DEFINE_LAUNCH(64, 2, false, true)
FA_DEFINE_LAUNCH(64, 3, false, true)
FA_DEFINE_LAUNCH(64, 4, false, true)
FA_DEFINE_LAUNCH(64, 2, true, true)
FA_DEFINE_LAUNCH(64, 3, true, true)
FA_DEFINE_LAUNCH(64, 4, true, true)
}  // namespace fa
