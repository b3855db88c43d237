// Dataflow-synchronised persistent decode kernel for sm_103a: n decode steps
// of one sequence in one cooperative launch, one CTA per SM.
//
// Phases and work split follow step.cuh (split-K by R input ranges, the
// o-projection's input build runs the attention of its range's kv heads), but
// no phase ends in a grid barrier. Every GEMV output travels as 64-bit words
// (value, flag) where the flag is the launch-wide step number: a consumer
// polls exactly the words it gathers, and a word is valid once its flag
// matches, so the data carries its own readiness and no fence, counter or
// second round trip sits between a producer's store and a consumer's use.
// Each phase owns its output words, so within a step nothing is overwritten;
// across steps the greedy choice (every CTA reads every CTA's candidate) is a
// complete exchange, and one release/acquire fence pair around it orders the
// KV-cache appends of a step before the next step's attention reads them.
//
// The producer warp walks the same (step, phase) sequence and streams the
// CTA's weight units through a ring of shared-memory slots with 1-D bulk
// copies; a slot is released unit by unit as consumer warps finish with it,
// so phases larger than the ring stream through it and the producer runs
// ahead across phase and step boundaries.
//
// The 4-bit unit dot is exact within its 64-input group: the build renders
// the group of x as 32-bit fixed point with one exponent (x = X * 2^e, every
// element of magnitude >= 2^-6 of the group's largest exact, the rest within
// 2^-31 of it), split into four byte limbs; dp4a multiplies them with the
// codes in integer arithmetic, the limb sums combine exactly in 64-bit
// integers, and one rounding to fp32 gives sum_j q_j x_j. The dequantisation
// s * that + m * sum_j x_j and the sum over groups are fp32.
#pragma once
#include "step.cuh"

#ifndef LLMQ_INFLIGHT
#define LLMQ_INFLIGHT 9
#endif
constexpr uint32_t kLInFlight = LLMQ_INFLIGHT;
#ifndef LLMQ_POLL_NS
#define LLMQ_POLL_NS 0  // pause between polling rounds of a gather (ns)
#endif

namespace llmq {

constexpr int kLWarps = 15;                       // consumer warps (480 threads, as the attention item expects)
constexpr int kLCThreads = kLWarps * 32;
constexpr int kLThreads = kLCThreads + 32;        // + one producer warp
constexpr int kLSlotBytes = 16384;                // 14 4-bit units or 16 bf16 units
constexpr int kLSlotUnits = 16;                   // unit credits of a slot's empty barrier
constexpr int kLNSlot = 9;
constexpr int kLRing = kLNSlot * kLSlotBytes;
constexpr int kLMaxKr = 4096;                     // widest per-CTA GEMV input
constexpr int kLMaxV = (kLMaxKr / 4 + kLCThreads - 1) / kLCThreads;  // float4s of it per thread
constexpr int kLRed = 320;                        // (tile, group block) partials of a phase (fits in the attention's shared memory)
constexpr int kLMaxRes = 1024;                    // residual range kept in shared memory
constexpr int kLMaxCTAs = 256;
constexpr int kLStampSteps = 8;                  // steps a profiled launch may time

enum LInMode : int { LIN_EMBED_F32 = 0, LIN_EMBED_BF16 = 1, LIN_RESID = 2, LIN_SWIGLU = 3, LIN_ATTN = 4, LIN_FINAL = 5 };

struct LPhase {
  int layer;
  const uint8_t* units;    // [n_rt][G] units
  int n_rt, G, K, bf16, unit_bytes;
  int R, GR, NB;           // input ranges, groups per range, group blocks per row tile
  int in_mode;
  const uint64_t* in_ll;   // partial words of the GEMV this build reads: [tile][in_R][32]
  int in_R;
  const uint64_t* res_ll;  // LIN_FINAL: the residual before the last down projection [dim]
  uint64_t* res_out;       // publish this build's residual range (the last layer's gate|up build)
  uint64_t* out_ll;        // [n_rt][R][32]; null for the LM head (its rows are whole logits)
  const float* norm_w;     // RMSNorm weight of this GEMV's input, or null
  uint64_t* ss_out;        // [4] sums of squares of the pre-norm input, one word per range
  const uint64_t* ss_in;   // [4] the sums of the GEMV whose outputs this build reads
  float* in_store;         // hidden-state capture of the (pre-norm) input, or null
  const float* q_norm;     // LIN_ATTN: per-head q/k RMSNorm weights (Qwen3), or null
  const float* k_norm;
};

struct StepLLParams {
  const LPhase* phases;    // the GEMV phases of one step, the LM head last
  int n_phases;
  int n_steps;
  int n_forced;            // steps whose input token is forced[s] (prompt tokens); then the greedy choice
  const int* forced;
  int dim, vocab;
  float eps;
  uint32_t* epoch;         // flag of this launch's first step; advanced by n_steps at the end
  int* abort;              // [1 + N]: abort word (zero before the launch), then each CTA's progress
  int* status;
  const void* embed;
  // attention
  int q_dim, kv_dim, Hkv, cap, rope_neox;
  const float2* rope;
  int* pos;                // position of step 0's token; advanced by n_steps at the end
  uint16_t* k_base;        // this sequence's cache [L][Hkv][cap][hd]
  uint16_t* v_base;
  size_t layer_stride;
  // greedy choice
  uint64_t* cand;          // [N][2] (value, index) words of every CTA's best logit
  float* logits;
  int* tok_io;             // step 0's token when n_forced == 0; the last choice at the end
  int* argmax_out;
  int* hist;
  int* hist_ctr;
  int hist_cap;
  unsigned long long* stamps;  // optional per (step, phase, CTA) records [.][16]
};

// ---- flagged words ----------------------------------------------------------
__device__ __forceinline__ uint64_t ll_pack(float v, uint32_t e) {
  return (static_cast<uint64_t>(e) << 32) | __float_as_uint(v);
}
__device__ __forceinline__ uint64_t ll_pack_i(int v, uint32_t e) {
  return (static_cast<uint64_t>(e) << 32) | static_cast<uint32_t>(v);
}
__device__ __forceinline__ float ll_val(uint64_t w) { return __uint_as_float(static_cast<uint32_t>(w)); }
__device__ __forceinline__ void ll_st(uint64_t* p, uint64_t w) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ void ll_st2(uint64_t* p, uint64_t a, uint64_t b) {
  asm volatile("st.relaxed.gpu.global.v2.b64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
// Two words (16-B aligned); zero (never a valid flag) when !pred.
__device__ __forceinline__ ulonglong2 ll_ld2(const uint64_t* p, bool pred = true) {
  ulonglong2 r;
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %3, 0;\n\tmov.b64 %0, 0;\n\tmov.b64 %1, 0;\n\t"
      "@q ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];\n\t}"
      : "=l"(r.x), "=l"(r.y)
      : "l"(p), "r"((uint32_t)pred)
      : "memory");
  return r;
}
__device__ __forceinline__ bool ll_ok(ulonglong2 w, uint32_t e) {
  return static_cast<uint32_t>(w.x >> 32) == e && static_cast<uint32_t>(w.y >> 32) == e;
}

// Gives up the wait when another CTA aborted or the wait limit passed (then
// aborts the launch itself).
// Waits are timed on the SM's cycle counter (reading %globaltimer costs about
// half a microsecond, which a wait would add to its own latency); the limit is
// 4e9 cycles, 2 s at 2 GHz. The abort word records where the first expired wait
// was (block, site). A normal wait lasts microseconds: the launch-wide abort
// flag (a global-memory read) is only consulted once a wait has run past 1e5
// cycles, so spinning warps put nothing on the memory system.
constexpr long long kWaitLimitCycles = 4000000000ll;
__device__ __forceinline__ long long lclock() { return clock64(); }
__device__ __forceinline__ bool ll_keep_waiting(const StepLLParams& sp, long long t0, unsigned it, int site) {
  if ((it & 15) != 0) return true;
  const long long dt = lclock() - t0;
  if (dt < 100000ll) return true;
  if (*(volatile int*)sp.abort) return false;
  if (dt > kWaitLimitCycles) {
    atomicOr(sp.status, ST_TIMEOUT);
    atomicCAS(sp.abort, 0, 1 + ((int)blockIdx.x << 8) + site);
    atomicCAS(sp.abort, 0, 1);
    return false;
  }
  return true;
}

// Gather NL pairs of words at addr(j) (valid where bit j of `mask` is set)
// until every one carries flag e; each round re-reads every pending pair (all
// loads of a round go out together: one round trip per round). Measured on
// GB300 against a probe-one-then-reload and a one-warp-sample-then-gather
// scheme, this full polling gives the shortest exchange (1.35 us per all-to-all
// of 16 KB per CTA idle, 1.74 us under a full weight stream).
template <int NL, typename Addr>
__device__ __forceinline__ bool ll_gather(ulonglong2 (&w)[NL], Addr addr, uint32_t mask, uint32_t e,
                                          const StepLLParams& sp, int site = 0) {
#pragma unroll
  for (int j = 0; j < NL; ++j) w[j] = ll_ld2(addr(j), (mask >> j) & 1u);
  uint32_t pend = 0;
#pragma unroll
  for (int j = 0; j < NL; ++j)
    if (((mask >> j) & 1u) && !ll_ok(w[j], e)) pend |= 1u << j;
  if (pend == 0) return true;
  const long long t0 = lclock();
  for (unsigned it = 1;; ++it) {
#pragma unroll
    for (int j = 0; j < NL; ++j)
      if ((pend >> j) & 1u) w[j] = ll_ld2(addr(j));
    uint32_t np = 0;
#pragma unroll
    for (int j = 0; j < NL; ++j)
      if (((pend >> j) & 1u) && !ll_ok(w[j], e)) np |= 1u << j;
    pend = np;
    if (pend == 0) return true;
    if (!ll_keep_waiting(sp, t0, it, site)) return false;
#if LLMQ_POLL_NS > 0
    __nanosleep(LLMQ_POLL_NS);
#endif
  }
}

// ---- shared memory ----------------------------------------------------------
template <int GQ, int HD>
struct LSmem {
  union {
    struct {
      union {
        uint4 xl[kLMaxKr / 4];  // 4-bit phases: [group][limb][4] limbs of X
        float xh[kLMaxKr];      // bf16 phases: the fp32 input
      } x;
      float fe[kLMaxKr / 64];   // 2^e / 16 per group
      float xs[kLMaxKr / 64];   // sum of the group's x
      float red[kLRed][32];     // (tile, group block) partials
    } g;
    StepAttnSmem<GQ, HD> a;
  } u;
  __align__(16) float xres[kLMaxRes];  // this CTA's range of the residual stream
  __align__(16) float fo[kSFuseOut];   // attention output of the o-projection range
  float wsum[kLWarps];
  float fbest[kLWarps];
  int ibest[kLWarps];
  float inv;      // 1/rms handed from the thread that read it
  int tok;        // the current step's input token
  LPhase ph[3];   // descriptors of the previous, current and next phase (a warp may still be
                  // publishing the previous phase while warp 0 fetches the next one)
  long long wstat[kLWarps][2];  // profiling: each warp's cycles waiting for units / in unit dots
  int flag_ok;    // the greedy-choice gather completed
  int abort;
  int issued;     // slot fills the producer issued (drain after an abort)
};

template <int GQ, int HD>
constexpr size_t stepll_smem_bytes() {
  return kLRing + ((sizeof(LSmem<GQ, HD>) + 15) & ~size_t(15)) + 2 * kLNSlot * sizeof(uint64_t);
}

__device__ __forceinline__ void mbar_arrive_cnt(uint64_t* bar, uint32_t n) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(n) : "memory");
}

// Bounded wait on a ring barrier; gives up on the launch's abort flag.
// The wait suspends the thread in hardware until the phase completes or the
// hinted time (20 us) passes, so a waiting warp takes no issue slots from the
// warps it shares a scheduler with.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 20000;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool lring_wait(uint64_t* bar, uint32_t parity, const StepLLParams& sp, int site) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = lclock();
  for (unsigned it = 1; !mbar_try_wait_sleep(bar, parity); ++it)
    if (!ll_keep_waiting(sp, t0, 16 * it, site)) return false;
  return true;
}
// A parity wait tells phases apart only one fill ahead: a consumer first waits
// until the producer has issued fill q of the ring (its slot's barrier then
// tracks that fill), then for the fill to land.
__device__ __forceinline__ bool lring_wait_fill(uint64_t* full, const volatile int* issued, uint32_t q,
                                                const StepLLParams& sp) {
  if ((uint32_t)*issued <= q) {
    const long long t0 = lclock();
    for (unsigned it = 1; (uint32_t)*issued <= q; ++it) {
      if (!ll_keep_waiting(sp, t0, it, 9)) return false;
      __nanosleep(64);  // the producer issues the fill once a slot frees up
    }
  }
  return lring_wait(&full[q % kLNSlot], (q / kLNSlot) & 1, sp, 2);
}

// This CTA's row tiles [t0, t1) and input range r of phase P.
struct LPart {
  int r, t0, t1;
  __device__ LPart(const LPhase& P, int c, int N) {
    const KRange kr(c, N, P.R);
    r = kr.r;
    t0 = kr.tile(c, P.n_rt);
    t1 = kr.tile(c + 1, P.n_rt);
  }
  __device__ bool first(int c, int N, int R) const { return c == KRange(c, N, R).c0; }
};

__device__ __forceinline__ int lslots(int U, int ub) {
  const int ups = kLSlotBytes / ub;
  return (U + ups - 1) / ups;
}

// ---- K/V rows of an attention item's first pass (see step_attn_prefetch) ----
template <int GQ, int HD>
__device__ void lattn_prefetch(const StepLLParams& sp, int layer, int g, int t1, int pos, StepAttnSmem<GQ, HD>& sa) {
  using SA = StepAttnSmem<GQ, HD>;
  constexpr int NT = kLCThreads, PP = SA::PP, CH = HD / 8;
  constexpr int TB = (2 * PP * CH + NT - 1) / NT;
  const int tid = threadIdx.x;
  const uint16_t* kc = sp.k_base + (size_t)layer * sp.layer_stride + (size_t)g * sp.cap * HD;
  const uint16_t* vc = sp.v_base + (size_t)layer * sp.layer_stride + (size_t)g * sp.cap * HD;
  const int n = min(PP, t1);
#pragma unroll
  for (int j = 0; j < TB; ++j) {
    const int idx = tid + j * NT, kv = idx / (PP * CH), rem = idx - kv * (PP * CH), row = rem / CH, ch = rem - row * CH;
    if (kv < 2 && row < n && row != pos)
      cp_async16(&(kv ? sa.vt : sa.kt)[row][8 * ch], (kv ? vc : kc) + (size_t)row * HD + 8 * ch);
  }
}

// ---- one kv head's attention over the whole cache (positions 0..pos), run
// by the consumer warps inside the o-projection's input build. q (GQ heads),
// k and v of the head come from the q|k|v partial words; `append`: this CTA
// writes the step's k, v into the cache. Output: fo[h * HD + d], normalised.
template <int GQ, int HD>
__device__ bool lattn_item(const StepLLParams& sp, const LPhase& P, int g, int pos, uint32_t E,
                           StepAttnSmem<GQ, HD>& sa, float* s_inv, bool append, float* fo, bool prefetched) {
  using SA = StepAttnSmem<GQ, HD>;
  constexpr int NT = kLCThreads, PP = SA::PP, RS = SA::RS, CH = HD / 8;
  constexpr int TB = (2 * PP * CH + NT - 1) / NT;
  static_assert((GQ + 1) * (HD / 2) + HD <= NT && GQ <= 8 && SA::NBW <= kLWarps && (GQ + 2) * HD / 2 < NT,
                "one RoPE pair or v element per thread, one q|k|v row pair per thread");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int len = pos + 1, t1 = len;
  uint16_t* kc = sp.k_base + (size_t)P.layer * sp.layer_stride + (size_t)g * sp.cap * HD;
  uint16_t* vc = sp.v_base + (size_t)P.layer * sp.layer_stride + (size_t)g * sp.cap * HD;
  if (!prefetched) lattn_prefetch<GQ, HD>(sp, P.layer, g, t1, pos, sa);

  constexpr int DPL = HD / 32;
  const int nrope = (GQ + 1) * (HD / 2);
  float2 rcs = make_float2(1.f, 0.f);
  if (tid < nrope) rcs = __ldg(sp.rope + (size_t)pos * (HD / 2) + tid % (HD / 2));
  float wn[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e)
    wn[e] = (P.q_norm && warp <= GQ) ? __ldg((warp < GQ ? P.q_norm : P.k_norm) + lane + 32 * e) : 1.f;

  // ---- q (GQ heads), k, v of this kv head: one row pair per thread, summed
  // over the input ranges' partial words; the last thread reads the norm's sums
  bool ok = true;
  {
    const int R = P.in_R;
    const int rr = 2 * tid;
    const bool act = rr < (GQ + 2) * HD;
    int row = 0;
    if (act)
      row = rr < GQ * HD ? g * GQ * HD + rr
                         : (rr < (GQ + 1) * HD ? sp.q_dim + g * HD + rr - GQ * HD
                                               : sp.q_dim + sp.kv_dim + g * HD + rr - (GQ + 1) * HD);
    const uint64_t* base = P.in_ll + ((size_t)(row >> 5) * R) * 32 + (row & 31);
    ulonglong2 w[4];
    ok = ll_gather<4>(w, [&](int j) { return base + j * 32; }, act ? (1u << R) - 1u : 0u, E, sp, 3);
    if (act) {
      float a = 0.f, b = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j < R) {
          a += ll_val(w[j].x);
          b += ll_val(w[j].y);
        }
      sa.cur[rr / HD][rr % HD] = a;
      sa.cur[rr / HD][rr % HD + 1] = b;
    }
    if (tid == NT - 1) {
      ulonglong2 s2[2];
      const bool ok2 = ll_gather<2>(s2, [&](int j) { return P.ss_in + 2 * j; }, 3u, E, sp, 4);
      ok = ok && ok2;
      *s_inv = rms_inv(make_float4(ll_val(s2[0].x), ll_val(s2[0].y), ll_val(s2[1].x), ll_val(s2[1].y)), sp.dim,
                       sp.eps);
    }
  }
  {
    // the first pass's rows: bf16 -> fp16 in place, zero rows up to a multiple of 16
    cp_async_wait_all();
    const int n = min(PP, t1), rows = ((n + 15) / 16) * 16;
#pragma unroll
    for (int j = 0; j < TB; ++j) {
      const int idx = tid + j * NT, kv = idx / (PP * CH), rem = idx - kv * (PP * CH), row = rem / CH, ch = rem - row * CH;
      if (kv < 2 && row < rows && row != pos) {
        uint4* q = reinterpret_cast<uint4*>(&(kv ? sa.vt : sa.kt)[row][8 * ch]);
        const uint4 w = row < n ? *q : make_uint4(0u, 0u, 0u, 0u);
        *q = make_uint4(bf16x2_to_f16x2(w.x), bf16x2_to_f16x2(w.y), bf16x2_to_f16x2(w.z), bf16x2_to_f16x2(w.w));
      }
    }
  }
  if (!consumer_and(ok)) return false;
  {
    const float inv = *s_inv;
    for (int i = tid; i < (GQ + 2) * HD; i += NT) (&sa.cur[0][0])[i] *= inv;
  }
  ConsumerSync::sync();
  if (P.q_norm) {
    if (warp <= GQ) {
      float* v = sa.cur[warp];
      float x[DPL], ss = 0.f;
#pragma unroll
      for (int e = 0; e < DPL; ++e) {
        x[e] = v[lane + 32 * e];
        ss += x[e] * x[e];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float inv = 1.0f / sqrtf(ss / (float)HD + sp.eps);
#pragma unroll
      for (int e = 0; e < DPL; ++e) v[lane + 32 * e] = x[e] * inv * wn[e];
    }
    ConsumerSync::sync();
  }
  // ---- RoPE at `pos`; q scaled by log2(e)/sqrt(hd); k, v rounded to bf16
  const float qscale = 1.4426950408889634f / sqrtf((float)HD);
  const bool owner = pos < PP;
  auto keep = [&](int r, int d, float x) {
    const __nv_bfloat16 b = __float2bfloat16_rn(x);
    const float xr = __bfloat162float(b);
    sa.cur[r][d] = xr;
    if (append) (r == GQ ? kc : vc)[(size_t)pos * HD + d] = __bfloat16_as_ushort(b);
    if (owner) (r == GQ ? sa.kt : sa.vt)[pos][d] = __half_as_ushort(__float2half_rn(xr));
  };
  if (tid < nrope) {
    const int h = tid / (HD / 2), i = tid % (HD / 2);
    float* v = sa.cur[h];
    const int ia = sp.rope_neox ? i : 2 * i, ib = sp.rope_neox ? i + HD / 2 : 2 * i + 1;
    const float x0 = v[ia], x1 = v[ib];
    const float y0 = x0 * rcs.x - x1 * rcs.y, y1 = x0 * rcs.y + x1 * rcs.x;
    if (h < GQ) {
      v[ia] = y0 * qscale;
      v[ib] = y1 * qscale;
    } else {
      keep(GQ, ia, y0);
      keep(GQ, ib, y1);
    }
  } else if (tid < nrope + HD) {
    keep(GQ + 1, tid - nrope, sa.cur[GQ + 1][tid - nrope]);
  }
  for (int i = tid; i < GQ * HD; i += NT) sa.acc[i / HD][i % HD] = 0.f;
  if (tid < GQ) {
    sa.accm[tid] = -INFINITY;
    sa.accl[tid] = 0.f;
  }
  ConsumerSync::sync();

  // ---- passes of PP positions: warp w scores positions 16w .. 16w+15 of all GQ heads
  uint4 tl[TB];
  for (int tp = 0; tp < t1; tp += PP) {
    const int n = min(PP, t1 - tp), nb = (n + 15) / 16;
    if (tp != 0) {
#pragma unroll
      for (int j = 0; j < TB; ++j) {
        const int idx = tid + j * NT, kv = idx / (PP * CH), rem = idx - kv * (PP * CH), row = rem / CH,
                  ch = rem - row * CH;
        const float4 v = ldcg4_if(reinterpret_cast<const float*>((kv ? vc : kc) + (size_t)(tp + row) * HD + 8 * ch),
                                  kv < 2 && row < n && tp + row != pos);
        tl[j] = make_uint4(__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z), __float_as_uint(v.w));
      }
      const int rows = ((n + 15) / 16) * 16;
#pragma unroll
      for (int j = 0; j < TB; ++j) {
        const int idx = tid + j * NT, kv = idx / (PP * CH), rem = idx - kv * (PP * CH), row = rem / CH,
                  ch = rem - row * CH;
        if (kv < 2 && row < rows && tp + row != pos)
          *reinterpret_cast<uint4*>(&(kv ? sa.vt : sa.kt)[row][8 * ch]) =
              make_uint4(bf16x2_to_f16x2(tl[j].x), bf16x2_to_f16x2(tl[j].y), bf16x2_to_f16x2(tl[j].z),
                         bf16x2_to_f16x2(tl[j].w));
      }
      if (pos >= tp && pos < tp + n)
        for (int d = tid; d < HD; d += NT) {
          sa.kt[pos - tp][d] = __half_as_ushort(__float2half_rn(sa.cur[GQ][d]));
          sa.vt[pos - tp][d] = __half_as_ushort(__float2half_rn(sa.cur[GQ + 1][d]));
        }
      ConsumerSync::sync();
    }
    if (warp < nb)
      attn_block16<GQ, HD, RS>(&sa.cur[0][0], &sa.kt[0][0], &sa.vt[0][0], 16 * warp, n - 16 * warp, lane,
                               &sa.tres[warp][0][0], HD + 2);
    ConsumerSync::sync();
    if (warp < GQ) {
      const int h = warp;
      const float am = sa.accm[h], al = sa.accl[h];
      const float mw = lane < nb ? sa.tres[lane][h][HD] : -INFINITY;
      const float lw = lane < nb ? sa.tres[lane][h][HD + 1] : 0.f;
      float M = fmaxf(mw, am);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      const float f = lane < nb ? exp2f(mw - M) : 0.f;
      float Lsum = lw * f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) Lsum += __shfl_xor_sync(0xffffffffu, Lsum, o);
      const float fa = am == -INFINITY ? 0.f : exp2f(am - M);
      __syncwarp();
      if (lane < SA::NBW) sa.fac[h][1 + lane] = f;
      if (lane == 0) {
        sa.fac[h][0] = fa;
        sa.accm[h] = M;
        sa.accl[h] = al * fa + Lsum;
      }
    }
    ConsumerSync::sync();
    for (int i = tid; i < GQ * HD; i += NT) {
      const int h = i / HD, d = i % HD;
      float O = sa.acc[h][d] * sa.fac[h][0];
#pragma unroll
      for (int w2 = 0; w2 < SA::NBW; ++w2)
        if (w2 < nb) O += sa.tres[w2][h][d] * sa.fac[h][1 + w2];
      sa.acc[h][d] = O;
    }
  }
  for (int i = tid; i < GQ * HD; i += NT) fo[i] = sa.acc[i / HD][i % HD] / sa.accl[i / HD];
  return true;
}

// ---- the kernel -------------------------------------------------------------
template <int GQ, int HD>
__global__ void __launch_bounds__(kLThreads, 1) stepll_kernel(const StepLLParams sp) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* ring = smem_raw;
  LSmem<GQ, HD>& sm = *reinterpret_cast<LSmem<GQ, HD>*>(smem_raw + kLRing);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + kLRing + ((sizeof(LSmem<GQ, HD>) + 15) & ~size_t(15)));
  uint64_t* empty = full + kLNSlot;

  const int c = blockIdx.x, N = gridDim.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kLNSlot; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kLSlotUnits);
    }
    mbar_fence_init();
    sm.abort = 0;
    sm.issued = 0;
  }
  __syncthreads();
  // profiling: (global time, SM cycles) at the start and the end map each
  // CTA's cycle stamps onto one time line
  if (sp.stamps && tid == 0) {
    sp.stamps[(size_t)c * 16 + 12] = globaltimer();
    sp.stamps[(size_t)c * 16 + 13] = clock64();
  }
  const uint32_t E0 = *reinterpret_cast<volatile uint32_t*>(sp.epoch);
  const int pos0 = *reinterpret_cast<volatile int*>(sp.pos);

  if (warp == kLWarps) {
    // ================= producer: the CTA's units of every GEMV phase of every step
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      uint32_t seq = 0;
      bool ok = true;
      for (int s = 0; s < sp.n_steps && ok; ++s)
        for (int ph = 0; ph < sp.n_phases && ok; ++ph) {
          // the descriptor's fields in registers: the copies' "memory" clobbers
          // would otherwise reload them from global memory for every slot
          const LPhase& P = sp.phases[ph];
          const LPart pt(P, c, N);
          const int GR = __ldg(&P.GR), UB = __ldg(&P.unit_bytes), G = __ldg(&P.G), ups = kLSlotBytes / UB;
          const uint8_t* units = reinterpret_cast<const uint8_t*>(__ldg(reinterpret_cast<const unsigned long long*>(&P.units)));
          const int U = (pt.t1 - pt.t0) * GR;
          const size_t row0 = (size_t)pt.t0 * G + (size_t)pt.r * GR;
          for (int u0 = 0; u0 < U; u0 += ups, ++seq) {
            const int si = seq % kLNSlot;
            if (seq >= kLNSlot && !lring_wait(&empty[si], ((seq / kLNSlot) - 1) & 1, sp, 1)) {
              ok = false;
              break;
            }
            // at most kLInFlight fills outstanding: deeper queues only add latency
            // to every other access in the memory system
            if (seq >= kLInFlight) {
              const uint32_t f = seq - kLInFlight;
              if (!lring_wait(&full[f % kLNSlot], (f / kLNSlot) & 1, sp, 8)) {
                ok = false;
                break;
              }
            }
            const int n = min(ups, U - u0);
            mbar_expect_tx(&full[si], n * UB);
            for (int v = u0; v < u0 + n;) {
              const int tl = v / GR, gp = v - tl * GR, run = min(u0 + n - v, GR - gp);
              bulk_g2s(ring + si * kLSlotBytes + (v - u0) * UB, units + (row0 + (size_t)tl * G + gp) * UB, run * UB,
                       &full[si], pol);
              v += run;
            }
            if (n < kLSlotUnits) mbar_arrive_cnt(&empty[si], kLSlotUnits - n);
            *(volatile int*)&sm.issued = seq + 1;
          }
        }
    }
  } else {
    // ================= consumers
    constexpr int NT = kLCThreads;
    uint32_t mlo, mhi;
    asm volatile("mov.b32 %0, 0x0F0F0F0F;" : "=r"(mlo));
    asm volatile("mov.b32 %0, 0xF0F0F0F0;" : "=r"(mhi));
    uint32_t seq = 0;  // slot fills consumed so far (mirrors the producer)
    bool ok = true;
    if (tid == 0) sm.tok = sp.n_forced > 0 ? __ldg(sp.forced) : *reinterpret_cast<volatile int*>(sp.tok_io);
    static_assert(sizeof(LPhase) % 4 == 0 && sizeof(LPhase) / 4 <= kLCThreads, "");
    // descriptor of the k-th phase of the launch: read into a register early,
    // stored into slot k % 3 late, so the load's latency never stalls a thread
    constexpr int kDescWords = (int)(sizeof(LPhase) / 4);
    auto desc_word = [&](int k) {
      return tid < kDescWords ? __ldg(reinterpret_cast<const int*>(&sp.phases[k % sp.n_phases]) + tid) : 0;
    };
    auto desc_store = [&](int k, int v) {
      if (tid < kDescWords) reinterpret_cast<int*>(&sm.ph[k % 3])[tid] = v;
    };
    desc_store(0, desc_word(0));
    ConsumerSync::sync();
    for (int s = 0; s < sp.n_steps && ok; ++s) {
      const uint32_t E = E0 + (uint32_t)s;
      const int pos = pos0 + s;
      const bool pos_ok = pos >= 0 && pos < sp.cap;
      if (!pos_ok && tid == 0 && c == 0) atomicOr(sp.status, ST_CTX_FULL);
      for (int ph = 0; ph < sp.n_phases && ok; ++ph) {
        const int kph = s * sp.n_phases + ph;
        const LPhase& P = sm.ph[kph % 3];
        const int next_desc = desc_word(kph + 1);  // stored after this phase's units
        auto progress = [&](int v) {  // where this CTA is (read by the host after a timeout)
          if (tid == 0) asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(sp.abort + 1 + c), "r"(v) : "memory");
        };
        progress(kph * 4);
        const LPart pt(P, c, N);
        const bool first = pt.first(c, N, P.R);
        const int Kr = P.K / P.R, n4 = Kr / 4;
        const int mode = P.in_mode;
        unsigned long long* st =
            sp.stamps ? sp.stamps + (((size_t)s * sp.n_phases + ph) * N + c) * 16 : nullptr;
        if (st && tid == 0) st[0] = clock64();

        // ---------------- input build
        // norm weights and, for the attention, the cached K/V rows do not depend on the step
        float4 w4[kLMaxV];
        float4 xv[kLMaxV];
        float ss = 0.f;
        if (mode == LIN_ATTN) {
          const int hpr = sp.Hkv / P.R;
          // the item's tiles share memory with the partial sums a slower warp
          // may still be publishing from the previous phase
          ConsumerSync::sync();
          if (pos_ok) {
            lattn_prefetch<GQ, HD>(sp, P.layer, pt.r * hpr, pos + 1, pos, sm.u.a);
            for (int j = 0; j < hpr && ok; ++j) {
              ok = lattn_item<GQ, HD>(sp, P, pt.r * hpr + j, pos, E, sm.u.a, &sm.inv, first, sm.fo + j * GQ * HD,
                                      j == 0);
              ConsumerSync::sync();  // the next item and the input build reuse the shared memory
            }
          }
#pragma unroll
          for (int j = 0; j < kLMaxV; ++j) {
            const int i = tid + j * NT;
            xv[j] = (i < n4 && pos_ok) ? reinterpret_cast<const float4*>(sm.fo)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        } else if (mode == LIN_EMBED_F32 || mode == LIN_EMBED_BF16) {
          int t = sm.tok;
          if (t < 0 || t >= sp.vocab) {
            if (tid == 0) atomicOr(sp.status, ST_BAD_TOKEN);
            t = 0;
          }
#pragma unroll
          for (int j = 0; j < kLMaxV; ++j) {
            const int i = tid + j * NT;
            if (mode == LIN_EMBED_BF16) {
              xv[j] = make_float4(0.f, 0.f, 0.f, 0.f);
              if (i < n4) {
                const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(sp.embed) +
                                                                     (size_t)t * P.K + pt.r * Kr) + i);
                xv[j] = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                                    __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
              }
            } else {
              xv[j] = ldnc4_if(static_cast<const float*>(sp.embed) + (size_t)t * P.K + pt.r * Kr + 4 * i, i < n4);
            }
            if (i < n4) reinterpret_cast<float4*>(sm.xres)[i] = xv[j];
          }
        } else if (mode == LIN_RESID || mode == LIN_FINAL) {
          // x = residual + sum of the previous GEMV's range partials (rows 32t..32t+31 per tile)
          const int R = P.in_R;
#pragma unroll
          for (int j = 0; j < kLMaxV; ++j) {
            const int i = tid + j * NT;
            const bool act = i < n4;
            const int e = pt.r * Kr + 4 * i;
            const uint64_t* base = P.in_ll + ((size_t)(e >> 5) * R) * 32 + (e & 31);
            const uint64_t* rb = P.res_ll + e;
            ulonglong2 w[10];
            const uint32_t mask = act ? (((1u << (2 * R)) - 1u) | (mode == LIN_FINAL ? 0x300u : 0u)) : 0u;
            ok = ll_gather<10>(w, [&](int k) { return k < 8 ? base + (k >> 1) * 32 + 2 * (k & 1) : rb + 2 * (k - 8); },
                               mask, E, sp, 5) && ok;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (k < R) {
                v.x += ll_val(w[2 * k].x);
                v.y += ll_val(w[2 * k].y);
                v.z += ll_val(w[2 * k + 1].x);
                v.w += ll_val(w[2 * k + 1].y);
              }
            float4 b;
            if (mode == LIN_FINAL) {
              b = make_float4(ll_val(w[8].x), ll_val(w[8].y), ll_val(w[9].x), ll_val(w[9].y));
            } else {
              b = act ? reinterpret_cast<const float4*>(sm.xres)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            xv[j] = make_float4(b.x + v.x, b.y + v.y, b.z + v.z, b.w + v.w);
            if (act && mode == LIN_RESID) reinterpret_cast<float4*>(sm.xres)[i] = xv[j];
            if (act && P.res_out && first)
              ll_st2(P.res_out + e, ll_pack(xv[j].x, E), ll_pack(xv[j].y, E)),
                  ll_st2(P.res_out + e + 2, ll_pack(xv[j].z, E), ll_pack(xv[j].w, E));
          }
        } else {  // LIN_SWIGLU
          // tile t of the gate|up GEMV: 16 gate rows, then their 16 up rows -> inputs 16t..16t+15
          const int R = P.in_R;
#pragma unroll
          for (int j = 0; j < kLMaxV; ++j) {
            const int i = tid + j * NT;
            const bool act = i < n4;
            const int f = pt.r * Kr + 4 * i, sub = f & 15;
            const uint64_t* base = P.in_ll + ((size_t)(f >> 4) * R) * 32 + sub;
            ulonglong2 w[16];
            ok = ll_gather<16>(w, [&](int k) { return base + (k >> 2) * 32 + ((k >> 1) & 1) * 16 + 2 * (k & 1); },
                               act ? (1u << (4 * R)) - 1u : 0u, E, sp, 6) && ok;
            float4 gt = make_float4(0.f, 0.f, 0.f, 0.f), up = gt;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              if (k < R) {
                gt.x += ll_val(w[4 * k].x);
                gt.y += ll_val(w[4 * k].y);
                gt.z += ll_val(w[4 * k + 1].x);
                gt.w += ll_val(w[4 * k + 1].y);
                up.x += ll_val(w[4 * k + 2].x);
                up.y += ll_val(w[4 * k + 2].y);
                up.z += ll_val(w[4 * k + 3].x);
                up.w += ll_val(w[4 * k + 3].y);
              }
            xv[j] = gt;
            w4[j] = up;  // (no norm weight on this GEMV's input: the register is free)
          }
          if (tid == 0) {
            ulonglong2 s2[2];
            ok = ll_gather<2>(s2, [&](int j) { return P.ss_in + 2 * j; }, 3u, E, sp, 7) && ok;
            sm.inv = rms_inv(make_float4(ll_val(s2[0].x), ll_val(s2[0].y), ll_val(s2[1].x), ll_val(s2[1].y)),
                             sp.dim, sp.eps);
          }
          ConsumerSync::sync();
          const float inv = sm.inv;
#pragma unroll
          for (int j = 0; j < kLMaxV; ++j) {
            const float4 g = xv[j], u = w4[j];
            xv[j] = make_float4(silu_fast(g.x * inv) * (u.x * inv), silu_fast(g.y * inv) * (u.y * inv),
                                silu_fast(g.z * inv) * (u.z * inv), silu_fast(g.w * inv) * (u.w * inv));
          }
        }
        if (!consumer_and(ok)) {
          ok = false;
          break;
        }
        if (st && tid == 0) {
          st[1] = clock64();
        }
        if (P.norm_w) {
#pragma unroll
          for (int j = 0; j < kLMaxV; ++j) {
            const int i = tid + j * NT;
            w4[j] = ldnc4_if(P.norm_w + pt.r * Kr + 4 * i, i < n4);
          }
        }
        // pre-norm input: hidden-state capture, sum of squares, then x * w and the unit operands
        const bool bf = P.bf16 != 0;
#pragma unroll
        for (int j = 0; j < kLMaxV; ++j) {
          const int i = tid + j * NT;
          if (j * NT >= n4) break;  // uniform
          const bool act = i < n4;
          float4 x = act ? xv[j] : make_float4(0.f, 0.f, 0.f, 0.f);
          if (act && P.in_store && (first || mode == LIN_FINAL) && (mode != LIN_FINAL || c == 0))
            reinterpret_cast<float4*>(P.in_store + pt.r * Kr)[i] = x;
          if (P.norm_w) {
            ss += (x.x * x.x + x.y * x.y) + (x.z * x.z + x.w * x.w);
            const float4 w = w4[j];
            x = make_float4(x.x * w.x, x.y * w.y, x.z * w.z, x.w * w.w);
          }
          q4_build_group(x, i, act, bf, sm.u.g.x.xl, sm.u.g.x.xh, sm.u.g.fe, sm.u.g.xs);
        }
        if (P.norm_w) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
          if (lane == 0) sm.wsum[warp] = ss;
        }
        ConsumerSync::sync();
        float inv_final = 1.f;
        if (P.norm_w) {
          float t = 0.f;
#pragma unroll
          for (int w = 0; w < kLWarps; ++w) t += sm.wsum[w];
          if (mode == LIN_FINAL) inv_final = 1.0f / sqrtf(t / (float)sp.dim + sp.eps);
          else if (first && warp == kLWarps - 1 && lane < 4 && (lane == pt.r || (pt.r == 0 && lane >= P.R)))
            ll_st(P.ss_out + lane, ll_pack(lane == pt.r ? t : 0.f, E));  // readers add four words; ranges >= R are 0
        }
        progress(kph * 4 + 1);
        if (st && tid == 0) st[2] = clock64();

        // ---------------- units: items (tile, group block), then per-tile sums
        const int nt = pt.t1 - pt.t0, GR = P.GR, NB = P.NB, BS = GR / NB, UB = P.unit_bytes;
        const int ups = kLSlotBytes / UB;
        const int n_items = nt * NB;
        long long t_wait = 0, t_dot = 0;
        // items go to the four schedulers in turn (warp w runs on scheduler w % 4;
        // scheduler 3 also hosts the producer and has three consumer warps), and
        // within a scheduler to its warps in turn; each warp takes its items in
        // increasing order, as the ring's progress needs
        const int smsp = warp & 3, kw = warp >> 2, nws = (kLWarps - smsp + 3) >> 2;
        for (int m = 0; ok; ++m) {
          const int it = smsp + 4 * (kw + nws * m);
          if (it >= n_items) break;
          const int tl = it / NB, gb = it - tl * NB;
          const int u0 = tl * GR + gb * BS;
          uint32_t q = seq + (uint32_t)(u0 / ups);  // ring fill of the unit, and its place in the fill
          int r = u0 - (u0 / ups) * ups;
          float acc = 0.f;
          for (int jb = 0; jb < BS; ++jb) {
            const int g = gb * BS + jb;
            const int si = q % kLNSlot;
            const long long ta = st ? clock64() : 0;
            if (!lring_wait_fill(full, &sm.issued, q, sp)) {
              ok = false;
              break;
            }
            const long long tb = st ? clock64() : 0;
            const uint8_t* ub = ring + si * kLSlotBytes + r * UB;
            if (bf) acc += bf16_unit_dot(ub, sm.u.g.x.xh + g * kBF16UnitCols, lane);
            else acc += q4_unit_dot_limbs(ub, sm.u.g.x.xl + 16 * g, sm.u.g.fe[g], sm.u.g.xs[g], lane, mlo, mhi);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[si]);
            if (st) {
              const long long tc = clock64();
              t_wait += tb - ta;
              t_dot += tc - tb;
            }
            if (++r == ups) {
              r = 0;
              ++q;
            }
          }
          sm.u.g.red[it][lane] = acc;
        }
        if (st && lane == 0) {
          sm.wstat[warp][0] = t_wait;
          sm.wstat[warp][1] = t_dot;
        }
        seq += (uint32_t)lslots(nt * GR, UB);
        desc_store(kph + 1, next_desc);  // the barrier below orders it before the next phase's reads
        if (!consumer_and(ok)) {
          ok = false;
          break;
        }
        progress(kph * 4 + 2);
        if (st && tid == 0) {
          st[3] = clock64();
          long long mw = 0, md = 0, sw = 0, sd = 0;
          for (int w = 0; w < kLWarps; ++w) {
            mw = max(mw, sm.wstat[w][0]);
            md = max(md, sm.wstat[w][1]);
            sw += sm.wstat[w][0];
            sd += sm.wstat[w][1];
          }
          st[5] = mw;
          st[6] = md;
          st[7] = sw;
          st[8] = sd;
        }
        if (P.out_ll) {
          for (int tl = warp; tl < nt; tl += kLWarps) {
            float v = 0.f;
            for (int gb = 0; gb < NB; ++gb) v += sm.u.g.red[tl * NB + gb][lane];
            ll_st(P.out_ll + ((size_t)(pt.t0 + tl) * P.R + pt.r) * 32 + lane, ll_pack(v, E));
          }
          if (st && tid == 0) st[4] = clock64();
        } else {
          // ---------------- LM head: whole logits (final norm's 1/rms), greedy choice
          float bv = -INFINITY;
          int bi = 0x7fffffff;
          bool nan = false;
          for (int tl = warp; tl < nt; tl += kLWarps) {
            float v = 0.f;
            for (int gb = 0; gb < NB; ++gb) v += sm.u.g.red[tl * NB + gb][lane];
            v *= inv_final;
            const int row = (pt.t0 + tl) * 32 + lane;
            if (row < sp.vocab) {
              sp.logits[row] = v;
              if (v != v) nan = true;
              else if (better(v, row, bv, bi)) { bv = v; bi = row; }
            }
          }
          if (nan) atomicOr(sp.status, ST_NAN);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
          }
          if (lane == 0) {
            sm.fbest[warp] = bv;
            sm.ibest[warp] = bi;
          }
          ConsumerSync::sync();  // also: every logit, cache and hidden store of the step is issued
          if (tid == 0) {
            for (int w = 0; w < kLWarps; ++w)
              if (better(sm.fbest[w], sm.ibest[w], bv, bi)) { bv = sm.fbest[w]; bi = sm.ibest[w]; }
            asm volatile("fence.acq_rel.gpu;" ::: "memory");  // release this CTA's cache appends
            ll_st2(sp.cand + 2 * c, ll_pack(bv, E), ll_pack_i(bi, E));
          }
          // every CTA's candidate -> the choice (value desc., index asc.)
          if (warp == 0) {
            ulonglong2 w[kLMaxCTAs / 32];
            const bool ok2 = ll_gather<kLMaxCTAs / 32>(
                w, [&](int k) { return sp.cand + 2 * (lane + 32 * k); },
                [&] {
                  uint32_t m = 0;
                  for (int k = 0; k < kLMaxCTAs / 32; ++k)
                    if (lane + 32 * k < N) m |= 1u << k;
                  return m;
                }(),
                E, sp, 8);
            bv = -INFINITY;
            bi = 0x7fffffff;
#pragma unroll
            for (int k = 0; k < kLMaxCTAs / 32; ++k)
              if (lane + 32 * k < N) {
                const float v = ll_val(w[k].x);
                const int i = (int)(uint32_t)w[k].y;
                if (better(v, i, bv, bi)) { bv = v; bi = i; }
              }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
              const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
              if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
            }
            // acquire: the next step's attention reads the cache rows other CTAs appended
            asm volatile("fence.acq_rel.gpu;" ::: "memory");
            if (lane == 0) {
              if (bi < 0 || bi >= sp.vocab) bi = 0;  // every logit NaN (the status says so)
              sm.flag_ok = ok2;
              if (c == 0) {
                const int h = *sp.hist_ctr + s;
                if (h < sp.hist_cap) sp.hist[h] = bi;
                *sp.argmax_out = bi;
                *sp.tok_io = bi;
              }
              sm.tok = (s + 1 < sp.n_forced) ? __ldg(sp.forced + s + 1) : bi;
            }
          }
          ConsumerSync::sync();
          ok = ok && sm.flag_ok;
        }
      }
    }
    if (!ok) *(volatile int*)&sm.abort = 1;
  }
  __syncthreads();
  if (sm.abort) {
    // drain: wait (bounded) for the producer's copies still landing in the ring
    if (tid == kLWarps * 32) {
      const int issued = sm.issued;
      for (int i = max(0, issued - kLNSlot); i < issued; ++i) {
        const long long t0 = lclock();
        while (!mbar_try_wait(&full[i % kLNSlot], (i / kLNSlot) & 1) && lclock() - t0 < kWaitLimitCycles) {
        }
      }
    }
    return;
  }
  if (sp.stamps && tid == 0) {
    sp.stamps[(size_t)c * 16 + 14] = globaltimer();
    sp.stamps[(size_t)c * 16 + 15] = clock64();
  }
  if (c == 0 && tid == 0) {
    *sp.epoch = E0 + (uint32_t)sp.n_steps;
    *sp.pos = pos0 + sp.n_steps;
    *sp.hist_ctr = *sp.hist_ctr + sp.n_steps;
  }
}

// The flag-synchronised step kernel for a GQA group and head_dim (defined in
// stepll_kernels.cu); fn is null for an unsupported shape.
KernelRef stepll_kernel_ref(int gq, int hd);

}  // namespace llmq
