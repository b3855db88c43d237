// Instantiations of the grid-barrier persistent step kernel (step.cuh) for
// the bf16 K/V cache, a translation unit of their own so that the library's
// parts compile in parallel; step_kernel_ref picks among them and the int8
// K/V instantiations of step_kernels_kv8.cu.
#include "step.cuh"

namespace llmq {

KernelRef step_kernel_ref_kv8(int gq, int hd, bool fused, bool w4a8);

template <int GQ, int HD>
KernelRef step_ref_t(bool fused, bool w4a8) {
  KernelRef r;
  r.smem = step_smem_bytes<GQ, HD>();
  if (fused)
    r.fn = w4a8 ? (const void*)step_kernel<GQ, HD, true, true, false> : (const void*)step_kernel<GQ, HD, true, false, false>;
  else
    r.fn = w4a8 ? (const void*)step_kernel<GQ, HD, false, true, false> : (const void*)step_kernel<GQ, HD, false, false, false>;
  return r;
}

KernelRef step_kernel_ref(int gq, int hd, bool fused, bool w4a8, bool kv8) {
  if (kv8) return step_kernel_ref_kv8(gq, hd, fused, w4a8);
  if (gq == 2 && hd == 64) return step_ref_t<2, 64>(fused, w4a8);
  if (gq == 8 && hd == 64) return step_ref_t<8, 64>(fused, w4a8);
  if (gq == 2 && hd == 128) return step_ref_t<2, 128>(fused, w4a8);
  return KernelRef{};
}

}  // namespace llmq
