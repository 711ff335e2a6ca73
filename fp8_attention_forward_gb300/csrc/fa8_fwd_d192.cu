// Instantiations of the forward kernels for (d, dv) = (192, 128) and (192, 192).
#include "fa8_launch.h"
namespace fa8 {
FA8_DEFINE_PREFILL(192, 128)
FA8_DEFINE_FWD(192, 192)
FA8_DEFINE_DECODE(192, 128)
}  // namespace fa8
