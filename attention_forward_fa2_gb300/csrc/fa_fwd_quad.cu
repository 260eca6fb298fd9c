// Kernel instantiations of the quad-shuffle softmax form (row max and row sum
// reduced across the four threads of a quad; 128-key tiles, no mask).
#include "fa_launch.h"

namespace fa {
FA_DEFINE_LAUNCH_QUAD(128, 2, false)
FA_DEFINE_LAUNCH_QUAD(128, 2, true)
FA_DEFINE_LAUNCH_QUAD(64, 3, false)
FA_DEFINE_LAUNCH_QUAD(64, 3, true)
}  // namespace fa
