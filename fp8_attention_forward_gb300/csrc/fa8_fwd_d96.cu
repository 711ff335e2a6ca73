// Instantiations of the forward kernels for (d, dv) = (96, 96).
#include "fa8_launch.h"
namespace fa8 {
FA8_DEFINE_PREFILL(96, 96)
}  // namespace fa8
