// Instantiations of the forward kernels for (d, dv) = (64, 64).
#include "fa8_launch.h"
namespace fa8 {
FA8_DEFINE_PREFILL(64, 64)
}  // namespace fa8
