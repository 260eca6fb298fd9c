// Kernel instantiations for d_head = 128, no mask, key tile 128 (two K/V ring
// slots fit next to the two query tiles: 64 KiB + 2 x 64 KiB).
#include "fa_launch.h"

namespace fa {
FA_DEFINE_LAUNCH(128, 128, 2, false, false)
FA_DEFINE_LAUNCH(128, 128, 2, true, false)
}  // namespace fa
