// Instantiation of the forward kernel for (d, dv) = (256, 256).
#include "fa8_launch.h"
namespace fa8 {
FA8_DEFINE_FWD(256, 256)
FA8_DEFINE_DECODE(256, 256)
}  // namespace fa8
