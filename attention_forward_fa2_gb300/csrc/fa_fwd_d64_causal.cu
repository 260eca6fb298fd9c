// Kernel instantiations for d_head = 64 with the causal mask (key tile 128).
#include "fa_launch.h"

namespace fa {
FA_DEFINE_LAUNCH(64, 128, 2, false, true)
FA_DEFINE_LAUNCH(64, 128, 3, false, true)
FA_DEFINE_LAUNCH(64, 128, 4, false, true)
FA_DEFINE_LAUNCH(64, 128, 2, true, true)
FA_DEFINE_LAUNCH(64, 128, 3, true, true)
FA_DEFINE_LAUNCH(64, 128, 4, true, true)
}  // namespace fa
