// ATTN_OPT_EXP2_FMA instances (a share of the exponentials on the FMA pipe):
// bf16 d = 64 and 128, e4m3 d = 128
#include "attn_instance.cuh"
namespace wsattn {
int launch_exp2_fma(const LaunchArgs& a, int dtype) {
  if (dtype == 2 && a.d == 64) return launch_mask_xf<2, 64>(a);
  if (dtype == 2 && a.d == 128) return launch_mask_xf<2, 128>(a);
  if (dtype == 3 && a.d == 128) return launch_mask_xf<3, 128>(a);
  return kErrUnsupported;
}
}  // namespace wsattn
