// Instantiations of the flag-synchronised persistent step kernel (stepll.cuh),
// a translation unit of their own so that the library's parts compile in
// parallel.
#include "stepll.cuh"

namespace llmq {

template <int GQ, int HD>
KernelRef stepll_ref_t() {
  KernelRef r;
  r.fn = (const void*)stepll_kernel<GQ, HD>;
  r.smem = stepll_smem_bytes<GQ, HD>();
  return r;
}

KernelRef stepll_kernel_ref(int gq, int hd) {
  if (gq == 2 && hd == 64) return stepll_ref_t<2, 64>();
  if (gq == 8 && hd == 64) return stepll_ref_t<8, 64>();
  if (gq == 2 && hd == 128) return stepll_ref_t<2, 128>();
  return KernelRef{};
}

}  // namespace llmq
