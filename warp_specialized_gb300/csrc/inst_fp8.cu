// e4m3 instances: d = 128
#include "attn_instance.cuh"
namespace wsattn {
int launch_fp8(const LaunchArgs& a) {
  switch (a.d) {
    case 128: return launch_mask<3, 128>(a);
    default: return kErrUnsupported;
  }
}
}  // namespace wsattn
