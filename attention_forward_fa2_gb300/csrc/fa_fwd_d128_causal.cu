// Kernel instantiations for d_head = 128 with the causal mask (key tile 128).
#include "fa_launch.h"

namespace fa {
FA_DEFINE_LAUNCH(128, 128, 2, false, true)
FA_DEFINE_LAUNCH(128, 128, 2, true, true)
}  // namespace fa
