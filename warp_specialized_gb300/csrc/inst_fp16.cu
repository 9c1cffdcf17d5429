// fp16 instances: d = 64, 128, 256
#include "attn_instance.cuh"
namespace wsattn {
int launch_fp16(const LaunchArgs& a) {
  switch (a.d) {
    case 64: return launch_mask<1, 64>(a);
    case 128: return launch_mask<1, 128>(a);
    case 256: return launch_mask<1, 256>(a);
    default: return kErrUnsupported;
  }
}
}  // namespace wsattn
