// fp32 instantiations of the split-K attention (see k_attn.cuh).
#include "k_attn.cuh"

namespace nosa {
cudaError_t launch_attention_f32(const Shape& s, const AttnArgs& a, int stages, int bps,
                                  int warps, cudaStream_t stream) {
  if (s.d == 64) return launch_attn_dispatch_w<float, 64>(s, a, stages, bps, warps, stream);
  if (s.d == 128) return launch_attn_dispatch_w<float, 128>(s, a, stages, bps, warps, stream);
  return cudaErrorInvalidValue;
}
int attention_occupancy_f32(const Shape& s, int stages, int bps, int warps) {
  if (s.d == 64) return attn_occupancy_dispatch_w<float, 64>(s, stages, bps, warps);
  if (s.d == 128) return attn_occupancy_dispatch_w<float, 128>(s, stages, bps, warps);
  return 0;
}
int attention_streamk_occupancy_f32(const Shape& s, int stages, int bps, int warps) {
  if (s.d == 64) return attn_streamk_occupancy_dispatch_w<float, 64>(s, stages, bps, warps);
  if (s.d == 128) return attn_streamk_occupancy_dispatch_w<float, 128>(s, stages, bps, warps);
  return 0;
}
}  // namespace nosa
