// Instantiations of the forward kernels for (d, dv) = (128, 128).
#include "fa8_launch.h"
namespace fa8 {
FA8_DEFINE_PREFILL(128, 128)
FA8_DEFINE_DECODE(128, 128)
}  // namespace fa8
