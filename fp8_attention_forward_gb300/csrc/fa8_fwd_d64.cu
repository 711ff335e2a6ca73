// Instantiation of the forward kernel for (d, dv) = (64, 64).
#include "fa8_launch.h"
namespace fa8 {
FA8_DEFINE_FWD(64, 64)
}  // namespace fa8
