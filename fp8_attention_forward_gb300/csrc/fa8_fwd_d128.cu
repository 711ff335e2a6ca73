// Instantiation of the forward kernel for (d, dv) = (128, 128).
#include "fa8_launch.h"
namespace fa8 {
FA8_DEFINE_FWD(128, 128)
FA8_DEFINE_DECODE(128, 128)
}  // namespace fa8
