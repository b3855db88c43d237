// Instantiations of the grid-barrier persistent step kernel (step.cuh) for
// the grouped int8 K/V cache, a translation unit of their own so that the
// library's parts compile in parallel.
#include "step.cuh"

namespace llmq {

template <int GQ, int HD>
KernelRef step_ref_kv8_t(bool fused, bool w4a8) {
  KernelRef r;
  r.smem = step_smem_bytes<GQ, HD>();
  if (fused)
    r.fn = w4a8 ? (const void*)step_kernel<GQ, HD, true, true, true> : (const void*)step_kernel<GQ, HD, true, false, true>;
  else
    r.fn = w4a8 ? (const void*)step_kernel<GQ, HD, false, true, true> : (const void*)step_kernel<GQ, HD, false, false, true>;
  return r;
}

KernelRef step_kernel_ref_kv8(int gq, int hd, bool fused, bool w4a8) {
  if (gq == 2 && hd == 64) return step_ref_kv8_t<2, 64>(fused, w4a8);
  if (gq == 8 && hd == 64) return step_ref_kv8_t<8, 64>(fused, w4a8);
  if (gq == 2 && hd == 128) return step_ref_kv8_t<2, 128>(fused, w4a8);
  return KernelRef{};
}

}  // namespace llmq
