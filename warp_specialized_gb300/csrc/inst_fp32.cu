// fp32 instances (tf32 matrix products): d = 64, 128
#include "attn_instance.cuh"
namespace wsattn {
int launch_fp32(const LaunchArgs& a) {
  switch (a.d) {
    case 64: return launch_mask<0, 64>(a);
    case 128: return launch_mask<0, 128>(a);
    default: return kErrUnsupported;
  }
}
}  // namespace wsattn
