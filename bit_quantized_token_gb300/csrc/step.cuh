// Persistent decode-step kernel for sm_103a: the whole batch-1 step in one
// cooperative launch, one CTA per SM.
//
// A step is a list of phases (per layer: q|k|v GEMV, attention, o GEMV,
// gate|up GEMV, down GEMV; then the LM-head GEMV and the logit reduction with
// the greedy choice). Between phases the consumer warps of every CTA meet at a
// software grid barrier (an arrival counter, bounded wait). The producer warp
// of each CTA never waits at those barriers: it walks the same phase list and
// streams the CTA's weight units of every GEMV phase, in order, through one
// shared-memory ring, so the weights of the next phases are already arriving
// while the current phase finishes and the barrier resolves.
//
// Split-K across CTAs leaves one partial sum per CTA that touches a row tile
// (S = 1, 2 or 4 slots per tile, unused slots zero); the next phase adds the
// slots while it builds its input vector (residual add, SwiGLU, RMSNorm are
// fused there), so no phase needs a fix-up of its own and no float atomics
// are used. Every input build issues all of its loads before it uses any of
// them: one L2 round trip per phase.
//
// Attention is flash-decoding over (kv head, split) items. An item loads its
// K/V rows into padded shared-memory tiles in the same round trip as its q|k|v
// gather; each warp then scores all GQ heads against 16 positions on the
// tensor cores (attn_mma.cuh) and the item leaves an unnormalised partial
// (o, max, sum) per split;
// with few splits the o-projection's input build merges them, so the merge
// costs no round trip of its own. With many splits (long caches) the last
// split of a kv head merges them instead.
#pragma once
#include "kernels.cuh"
#include "attn_mma.cuh"

namespace llmq {

// 15 consumer warps + 1 producer warp = 4 warps per scheduler, 128 registers each
constexpr int kSWarps = 15;                      // consumer warps
constexpr int kSCThreads = kSWarps * 32;         // consumer threads
constexpr int kSThreads = kSCThreads + 32;       // + one producer warp
constexpr int kSChunk = kSWarps;                 // units per ring slot: one per consumer warp
constexpr int kSSlot = kSChunk * kQ4UnitBytes;   // 17280 B (bf16 chunks use 15360 B)
constexpr int kSNSlot = 8;
constexpr int kSRing = kSNSlot * kSSlot;         // 138240 B
constexpr int kSRLoc = 6;                        // row tiles a reduction window may touch
constexpr int kSMaxV = (kMaxK / 4 + kSCThreads - 1) / kSCThreads;  // float4s of a K-vector per thread
constexpr int kSDefer = 4;                       // splits the o-projection's input build merges
constexpr int kSMaxDim = 4096;                   // widest residual stream (kept in shared memory)

// Cache positions staged per attention pass (the K/V tiles fill about 36 KB
// resp. 52 KB of shared memory); a split is one pass unless the split count
// is capped.
__host__ __device__ constexpr int step_attn_pp(int hd) { return hd == 64 ? 128 : 96; }
__host__ __device__ inline int step_splits(int len, int P, int hd) {
  const int s = (len + step_attn_pp(hd) - 1) / step_attn_pp(hd);
  return s < 1 ? 1 : (s < P ? s : P);
}

enum PhaseType : int { PH_GEMV = 0, PH_ATTN = 1, PH_LOGITS = 2 };
enum InMode : int { IN_EMBED_F32 = 0, IN_EMBED_BF16 = 1, IN_PLAIN = 2, IN_RESID = 3, IN_SWIGLU = 4, IN_ATTN = 5 };

struct Phase {
  int type;
  int layer;
  // ---- GEMV
  const uint8_t* units;
  int n_rt, G, K, bf16, unit_bytes;
  Part part;
  float* out_part;        // [n_rt][part.S][32], unused slots stay zero
  int in_mode;
  const float* in_base;   // IN_PLAIN: the vector; IN_RESID: the residual base
  const float* in_part;   // IN_RESID / IN_SWIGLU: partials of the previous GEMV
  int in_S;               // 1, 2 or 4
  float* in_store;        // CTA 0 stores the built (pre-norm) vector here, or null
  const float* norm_w;    // RMSNorm weight, or null
  // ---- ATTN
  const float* qkv_part;
  int qkv_S;
  const float* q_norm;
  const float* k_norm;
  // ---- LOGITS
  const float* lm_part;
  int lm_S, vocab;
};

struct StepParams {
  const Phase* phases;
  int n_phases;
  int* sync;              // [0] arrivals (phases x CTAs), [1] abort; zeroed before each launch
  int* status;
  const void* embed;
  const int* tok;
  int vocab;
  float eps;
  // attention
  int q_dim, kv_dim, Hkv, P, cap, rope_neox;
  const float2* rope;
  int* pos;               // position of the sequence (advanced by the greedy choice)
  uint16_t* k_base;       // layer 0 of this sequence's cache: [L][Hkv][cap][hd]
  uint16_t* v_base;
  size_t layer_stride;    // elements per layer of the cache
  float* attn_o;          // [Hkv][P][GQ][hd] unnormalised split outputs
  float* attn_ml;         // [Hkv][P][GQ][2] (max, sum) of the splits
  int* attn_cnt;          // [Hkv], zero between launches (merge by the last split)
  float* obuf;            // [q_dim] merged output when the last split merges
  // greedy choice
  float* logits;
  float* cand_v;
  int* cand_i;
  int* gcounter;
  int* tok_io;
  int* argmax_out;
  int* hist;
  int* hist_ctr;
  int hist_cap;
};

struct ConsumerSync {
  __device__ static void sync() { asm volatile("bar.sync 1, %0;" ::"n"(kSCThreads) : "memory"); }
};

// Consumer barrier that also ANDs a flag over the consumer threads.
__device__ __forceinline__ bool consumer_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kSCThreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Partial arrays are [tile][S][32] floats with S = 1 << lgS. Float4 f covers
// rows 4*(f & 7) .. +3 of slot (f >> 3) & (S-1) of tile f >> (3 + lgS); as 8S
// divides 32, the slots of a row quad sit in lanes l, l^8 (, l^16, l^24) of
// one warp and a butterfly adds them. Every lane ends with the full sum.
__device__ __forceinline__ float4 slot_sum(float4 a, int lgS) {
  if (lgS >= 1) {
    a.x += __shfl_xor_sync(0xffffffffu, a.x, 8);
    a.y += __shfl_xor_sync(0xffffffffu, a.y, 8);
    a.z += __shfl_xor_sync(0xffffffffu, a.z, 8);
    a.w += __shfl_xor_sync(0xffffffffu, a.w, 8);
  }
  if (lgS >= 2) {
    a.x += __shfl_xor_sync(0xffffffffu, a.x, 16);
    a.y += __shfl_xor_sync(0xffffffffu, a.y, 16);
    a.z += __shfl_xor_sync(0xffffffffu, a.z, 16);
    a.w += __shfl_xor_sync(0xffffffffu, a.w, 16);
  }
  return a;
}
__device__ __forceinline__ int log2_slots(int S) { return S >= 4 ? 2 : S >= 2 ? 1 : 0; }

// Consumer-side grid barrier: wait until `target` arrivals (bounded). Any
// timeout sets the shared abort flag, which ends every other wait at once.
__device__ bool grid_wait(const StepParams& sp, int target, int* s_flag) {
  if (threadIdx.x == 0) {
    int ok = 1;
    if (ld_acquire(sp.sync) < target) {
      const unsigned long long t0 = globaltimer();
      unsigned ns = 16;
      while (ld_acquire(sp.sync) < target) {
        if (*(volatile int*)(sp.sync + 1)) { ok = 0; break; }
        if (globaltimer() - t0 > kWaitLimitNs) {
          atomicOr(sp.status, ST_TIMEOUT);
          atomicExch(sp.sync + 1, 1);
          ok = 0;
          break;
        }
        __nanosleep(ns);
        ns = ns < 64 ? 2 * ns : 64;
      }
    }
    *s_flag = ok;
  }
  ConsumerSync::sync();
  return *s_flag != 0;
}

// The release add orders every consumer's earlier writes (they precede it
// through the CTA barrier) before the arrival; grid_wait's acquire load pairs
// with it.
__device__ __forceinline__ void grid_arrive(const StepParams& sp) {
  ConsumerSync::sync();
  if (threadIdx.x == 0) asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(sp.sync) : "memory");
}

// Bounded mbarrier wait that also gives up when another CTA aborted the step.
__device__ __forceinline__ bool ring_wait(uint64_t* bar, uint32_t parity, const StepParams& sp) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  unsigned ns = 32;
  while (!mbar_try_wait(bar, parity)) {
    if (*(volatile int*)(sp.sync + 1)) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      atomicOr(sp.status, ST_TIMEOUT);
      atomicExch(sp.sync + 1, 1);
      return false;
    }
    __nanosleep(ns);
    ns = ns < 256 ? 2 * ns : 256;
  }
  return true;
}

// Shared memory of one attention item.
template <int GQ, int HD>
struct StepAttnSmem {
  static constexpr int PP = step_attn_pp(HD);  // positions per pass
  static constexpr int RS = HD + 8;             // padded row (halves): conflict-free ldmatrix
  static constexpr int NBW = PP / 16;           // warps with a 16-position block
  uint16_t kt[PP][RS];        // staged K rows (fp16)
  uint16_t vt[PP][RS];
  float cur[GQ + 2][HD];      // this step's q heads (scaled after RoPE), k, v of the kv head
  float tres[NBW][GQ][HD + 2];  // per block warp and head: o, max, sum
  float acc[GQ][HD];          // running output of the item over its passes
  float accm[GQ], accl[GQ];
  float fac[GQ][NBW + 1];
  int is_last;
};

template <int GQ, int HD>
struct StepSmem {
  union {
    struct {
      float xh[kMaxK];                     // input vector of the GEMV
      float xs[kMaxK / 64];                // its per-group sums
      float red[kSRLoc][kSWarps][32];      // per-warp row-tile sums of a window
      float carry[2][32];
    } g;
    StepAttnSmem<GQ, HD> a;
    struct {
      float fbest[kSWarps];
      int ibest[kSWarps];
      int last;
    } l;
  } u;
  __align__(16) float xres[kSMaxDim];  // this CTA's copy of the residual stream (pre-norm)
  Phase ph[2];            // descriptors of the current and the next phase
  float bred[kSWarps];
  int carry_rt[2];
  int flag;
  int abort;
  int issued;
};

// ---------------------------------------------------------------------------
// One (kv head g, split) attention item, run by the consumer warps.
template <int GQ, int HD>
__device__ void step_attn_item(const StepParams& sp, const Phase& P, int g, int split, int P_eff, int pos,
                               StepAttnSmem<GQ, HD>& sa) {
  using SA = StepAttnSmem<GQ, HD>;
  constexpr int NT = kSCThreads, PP = SA::PP, RS = SA::RS, CH = HD / 8;
  constexpr int TB = (2 * PP * CH + NT - 1) / NT;  // 16-B tile loads per thread
  static_assert((GQ + 1) * (HD / 2) + HD <= NT && GQ <= 8 && SA::NBW <= kSWarps,
                "one RoPE pair or v element per thread, GQ <= 8");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int len = pos + 1;
  const int t0 = (int)((int64_t)len * split / P_eff), t1 = (int)((int64_t)len * (split + 1) / P_eff);
  uint16_t* kc = sp.k_base + (size_t)P.layer * sp.layer_stride + (size_t)g * sp.cap * HD;
  uint16_t* vc = sp.v_base + (size_t)P.layer * sp.layer_stride + (size_t)g * sp.cap * HD;

  // K/V rows tp .. tp+n-1 -> registers (zero beyond the split); stored into
  // the padded tiles once the previous readers are done
  uint4 tl[TB];
  auto load_tile = [&](int tp) {
    const int n = min(PP, t1 - tp);
#pragma unroll
    for (int j = 0; j < TB; ++j) {
      const int idx = tid + j * NT, kv = idx / (PP * CH), rem = idx - kv * (PP * CH), row = rem / CH, ch = rem - row * CH;
      const float4 v = ldcg4_if(reinterpret_cast<const float*>((kv ? vc : kc) + (size_t)(tp + row) * HD + 8 * ch),
                                kv < 2 && row < n);
      tl[j] = make_uint4(__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z), __float_as_uint(v.w));
    }
  };
  auto store_tile = [&](int tp) {
    const int rows = ((min(PP, t1 - tp) + 15) / 16) * 16;
#pragma unroll
    for (int j = 0; j < TB; ++j) {
      const int idx = tid + j * NT, kv = idx / (PP * CH), rem = idx - kv * (PP * CH), row = rem / CH, ch = rem - row * CH;
      if (kv < 2 && row < rows)
        *reinterpret_cast<uint4*>(&(kv ? sa.vt : sa.kt)[row][8 * ch]) =
            make_uint4(bf16x2_to_f16x2(tl[j].x), bf16x2_to_f16x2(tl[j].y), bf16x2_to_f16x2(tl[j].z),
                       bf16x2_to_f16x2(tl[j].w));
    }
  };
  load_tile(t0);

  // RoPE factors and q/k norm weights do not depend on the step: load them
  // in the same round trip as the q|k|v gather and the first tile
  constexpr int DPL = HD / 32;
  const int nrope = (GQ + 1) * (HD / 2);
  float2 rcs = make_float2(1.f, 0.f);
  if (tid < nrope) rcs = __ldg(sp.rope + (size_t)pos * (HD / 2) + tid % (HD / 2));
  float wn[DPL];
#pragma unroll
  for (int e = 0; e < DPL; ++e)
    wn[e] = (P.q_norm && warp <= GQ) ? __ldg((warp < GQ ? P.q_norm : P.k_norm) + lane + 32 * e) : 1.f;

  // ---- gather q (GQ heads), k and v of this kv head from the QKV partials
  {
    const int lg = log2_slots(P.qkv_S);
    const int nq = GQ * HD / 32, nk = HD / 32;
    const int qt0 = g * nq, kt0 = (sp.q_dim + g * HD) / 32, vt0 = (sp.q_dim + sp.kv_dim + g * HD) / 32;
    const int T4 = (nq + 2 * nk) << (3 + lg);
    constexpr int RB = ((GQ + 2) * HD / 32 * 4 * 8 + NT - 1) / NT;  // covers S <= 4 in one batch
    float4 a[RB];
#pragma unroll
    for (int j = 0; j < RB; ++j) {
      const int f = tid + j * NT;
      const int ti = f >> (3 + lg);
      const int tile = ti < nq ? qt0 + ti : (ti < nq + nk ? kt0 + ti - nq : vt0 + ti - nq - nk);
      a[j] = ldcg4_if(P.qkv_part + ((size_t)tile * (8 << lg) + (f & ((8 << lg) - 1))) * 4, f < T4);
    }
#pragma unroll
    for (int j = 0; j < RB; ++j) {
      const float4 v = slot_sum(a[j], lg);
      const int f = tid + j * NT;
      if (f < T4 && ((f >> 3) & ((1 << lg) - 1)) == 0)
        *reinterpret_cast<float4*>(&sa.cur[0][0] + (f >> (3 + lg)) * 32 + (f & 7) * 4) = v;
    }
  }
  store_tile(t0);
  ConsumerSync::sync();
  // ---- per-head RMSNorm of q and k (Qwen3): warp h < GQ takes q head h, warp GQ takes k
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
  // ---- RoPE at `pos` (pairs (2i, 2i+1) or (i, i + HD/2)) of the q heads and
  // k; q is then scaled by log2(e)/sqrt(hd), k and v are rounded to bf16
  // (the split owning `pos` appends them and puts them into its tile)
  const float qscale = 1.4426950408889634f / sqrtf((float)HD);
  const bool owner = split == P_eff - 1 && pos - t0 < PP;
  auto keep = [&](int r, int d, float x) {  // final value of cur[r][d], r >= GQ
    const __nv_bfloat16 b = __float2bfloat16_rn(x);
    const float xr = __bfloat162float(b);
    sa.cur[r][d] = xr;
    if (split == P_eff - 1) {
      (r == GQ ? kc : vc)[(size_t)pos * HD + d] = __bfloat16_as_ushort(b);
      if (owner) (r == GQ ? sa.kt : sa.vt)[pos - t0][d] = __half_as_ushort(__float2half_rn(xr));
    }
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

  // ---- passes of at most PP positions: warp w takes positions 16w .. 16w+15
  for (int tp = t0; tp < t1; tp += PP) {
    const int n = min(PP, t1 - tp), nb = (n + 15) / 16;
    if (tp != t0) {
      load_tile(tp);
      store_tile(tp);
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
    const size_t pbase = ((size_t)g * sp.P + split) * GQ;
    if (tp + PP >= t1) {
      // last pass: merge its warps with the running output into the split's partial
      for (int i = tid; i < GQ * HD; i += NT) {
        const int h = i / HD, d = i % HD;
        float M = sa.accm[h];
        for (int w = 0; w < nb; ++w) M = fmaxf(M, sa.tres[w][h][HD]);
        const float fa = sa.accm[h] == -INFINITY ? 0.f : exp2f(sa.accm[h] - M);
        float O = sa.acc[h][d] * fa, L = sa.accl[h] * fa;
        for (int w = 0; w < nb; ++w) {
          const float f = exp2f(sa.tres[w][h][HD] - M);
          O += sa.tres[w][h][d] * f;
          L += sa.tres[w][h][HD + 1] * f;
        }
        sp.attn_o[pbase * HD + i] = O;
        if (d == 0) {
          sp.attn_ml[(pbase + h) * 2] = M;
          sp.attn_ml[(pbase + h) * 2 + 1] = L;
        }
      }
      break;
    }
    // fold the pass into the running output
    if (tid < GQ) {
      const int h = tid;
      float M = sa.accm[h];
      for (int w = 0; w < nb; ++w) M = fmaxf(M, sa.tres[w][h][HD]);
      const float fa = sa.accm[h] == -INFINITY ? 0.f : exp2f(sa.accm[h] - M);
      float L = sa.accl[h] * fa;
      sa.fac[h][0] = fa;
      for (int w = 0; w < nb; ++w) {
        const float f = exp2f(sa.tres[w][h][HD] - M);
        sa.fac[h][1 + w] = f;
        L += sa.tres[w][h][HD + 1] * f;
      }
      sa.accm[h] = M;
      sa.accl[h] = L;
    }
    ConsumerSync::sync();
    for (int i = tid; i < GQ * HD; i += NT) {
      const int h = i / HD, d = i % HD;
      float O = sa.acc[h][d] * sa.fac[h][0];
      for (int w = 0; w < nb; ++w) O += sa.tres[w][h][d] * sa.fac[h][1 + w];
      sa.acc[h][d] = O;
    }
    ConsumerSync::sync();
  }

  // ---- the split's partial is written (last pass above)
  if (P_eff <= kSDefer) return;  // the o-projection's input build merges the splits
  // many splits: the last one of this kv head merges them into obuf
  __threadfence();
  ConsumerSync::sync();
  if (tid == 0) sa.is_last = (atomicAdd(&sp.attn_cnt[g], 1) == P_eff - 1);
  ConsumerSync::sync();
  if (sa.is_last) {
    __threadfence();
    const float* ho = sp.attn_o + (size_t)g * sp.P * GQ * HD;
    const float* hm = sp.attn_ml + (size_t)g * sp.P * GQ * 2;
    for (int i = tid; i < GQ * HD; i += NT) {
      const int h = i / HD, d = i % HD;
      float M = -INFINITY;
      for (int s = 0; s < P_eff; ++s) M = fmaxf(M, __ldcg(hm + ((size_t)s * GQ + h) * 2));
      float L = 0.f, O = 0.f;
      for (int s = 0; s < P_eff; ++s) {
        const float f = exp2f(__ldcg(hm + ((size_t)s * GQ + h) * 2) - M);
        L += __ldcg(hm + ((size_t)s * GQ + h) * 2 + 1) * f;
        O += __ldcg(ho + ((size_t)s * GQ + h) * HD + d) * f;
      }
      sp.obuf[(g * GQ + h) * HD + d] = O / L;
    }
    if (tid == 0) sp.attn_cnt[g] = 0;
  }
}

template <int GQ, int HD>
__global__ void __launch_bounds__(kSThreads, 1) step_kernel(const StepParams sp) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* ring = smem_raw;
  StepSmem<GQ, HD>& sm = *reinterpret_cast<StepSmem<GQ, HD>*>(smem_raw + kSRing);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem_raw + kSRing + ((sizeof(StepSmem<GQ, HD>) + 15) & ~size_t(15)));
  uint64_t* empty = full + kSNSlot;

  const int c = blockIdx.x, N = gridDim.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kSNSlot; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kSWarps);
    }
    mbar_fence_init();
    sm.abort = 0;
    sm.issued = 0;
  }
  __syncthreads();

  if (warp == kSWarps) {
    // ================= producer: every GEMV phase's units, in phase order
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int gi = 0;
      bool ok = true;
      for (int ph = 0; ph < sp.n_phases && ok; ++ph) {
        const Phase& P = sp.phases[ph];
        if (P.type != PH_GEMV || c >= P.part.N) continue;  // small GEMVs use the first part.N CTAs
        const int u0 = P.part.begin(c), u1 = P.part.begin(c + 1);
        for (int ub = u0; ub < u1; ub += kSChunk, ++gi) {
          const int s = gi % kSNSlot;
          if (gi >= kSNSlot && !ring_wait(&empty[s], ((gi / kSNSlot) - 1) & 1, sp)) {
            ok = false;
            break;
          }
          const int bytes = min(kSChunk, u1 - ub) * P.unit_bytes;
          mbar_expect_tx(&full[s], bytes);
          bulk_g2s(ring + s * kSSlot, P.units + (size_t)ub * P.unit_bytes, bytes, &full[s], pol);
          sm.issued = gi + 1;
        }
      }
    }
  } else {
    // ================= consumers
    constexpr int NT = kSCThreads;
    int gi = 0;
    // the position only changes at the very end of the step (greedy choice)
    const int spos = *sp.pos;
    // descriptors go to shared memory one phase ahead (the phase table is immutable)
    static_assert(sizeof(Phase) % 4 == 0, "");
    auto fetch_phase = [&](int ph) {
      if (ph < sp.n_phases)
        for (int i = tid; i < (int)(sizeof(Phase) / 4); i += NT)
          reinterpret_cast<int*>(&sm.ph[ph & 1])[i] = __ldg(reinterpret_cast<const int*>(&sp.phases[ph]) + i);
    };
    fetch_phase(0);
    ConsumerSync::sync();
    for (int ph = 0; ph < sp.n_phases; ++ph) {
      const Phase& P = sm.ph[ph & 1];
      // norm weights do not depend on the step: in flight while the barrier resolves
      float4 w4[kSMaxV];
      {
        const bool nw = P.type == PH_GEMV && P.norm_w != nullptr;
#pragma unroll
        for (int j = 0; j < kSMaxV; ++j) {
          const int i = tid + j * NT;
          w4[j] = ldnc4_if(nw ? P.norm_w + 4 * i : nullptr, nw && i < P.K / 4);
        }
      }
      // the unit range of this CTA (divisions: done while the barrier resolves)
      int u0 = 0, u1 = 0, n_chunks = 0, wch = 1, k_rt = 0, k_g = 0, rt0 = 0;
      if (P.type == PH_GEMV && c < P.part.N) {
        u0 = P.part.begin(c);
        u1 = P.part.begin(c + 1);
        rt0 = u0 / P.G;
        n_chunks = (u1 - u0 + kSChunk - 1) / kSChunk;
        wch = max(1, ((kSRLoc - 2) * P.G + 1) / kSChunk);
        k_rt = (u0 + warp) / P.G;
        k_g = (u0 + warp) - k_rt * P.G;
      }
      // the next descriptor goes to the buffer the previous phase used: its
      // round trip overlaps the barrier wait
      fetch_phase(ph + 1);
      if (ph > 0 && !grid_wait(sp, ph * N, &sm.flag)) {
        sm.abort = 1;
        break;
      }
      if (P.type == PH_GEMV) {
        // ---------------- build the input vector: every load of the build in one round trip
        const int K = P.K, n4 = K / 4;
        float4* xh4 = reinterpret_cast<float4*>(sm.u.g.xh);
        float ss = 0.f;
        float4* xr4 = reinterpret_cast<float4*>(sm.xres);
        auto put = [&](int i4, float4 v) {  // pre-norm inputs 4*i4 .. 4*i4+3
          xh4[i4] = v;
          if (P.in_store && c == 0) reinterpret_cast<float4*>(P.in_store)[i4] = v;
          ss += (v.x * v.x + v.y * v.y) + (v.z * v.z + v.w * v.w);
        };
        if (P.in_mode == IN_RESID) {
          // x = residual (this CTA's resident copy) + sum of the previous
          // GEMV's slots (row tiles of 32 inputs); x becomes the new residual
          constexpr int RB = 8;
          const int lg = log2_slots(P.in_S);
          const int T4 = (K / 32) << (3 + lg);
          for (int f0 = 0; f0 < T4; f0 += RB * NT) {
            float4 a[RB];
#pragma unroll
            for (int j = 0; j < RB; ++j) {
              const int f = f0 + tid + j * NT;
              a[j] = ldcg4_if(P.in_part + (size_t)f * 4, f < T4);
            }
#pragma unroll
            for (int j = 0; j < RB; ++j) {
              const float4 s = slot_sum(a[j], lg);
              const int f = f0 + tid + j * NT;
              if (f < T4 && ((f >> 3) & ((1 << lg) - 1)) == 0) {
                const int r4 = ((f >> (3 + lg)) << 3) + (f & 7);
                const float4 b = xr4[r4];
                const float4 x = make_float4(b.x + s.x, b.y + s.y, b.z + s.z, b.w + s.w);
                xr4[r4] = x;
                put(r4, x);
              }
            }
          }
        } else if (P.in_mode == IN_SWIGLU) {
          // row tile t of the gate|up GEMV: 16 gate rows, then their 16 up rows -> inputs 16t..16t+15
          constexpr int RB = 12;
          const int lg = log2_slots(P.in_S);
          const int T4 = (K / 16) << (3 + lg);
          for (int f0 = 0; f0 < T4; f0 += RB * NT) {
            float4 a[RB];
#pragma unroll
            for (int j = 0; j < RB; ++j) {
              const int f = f0 + tid + j * NT;
              a[j] = ldcg4_if(P.in_part + (size_t)f * 4, f < T4);
            }
#pragma unroll
            for (int j = 0; j < RB; ++j) {
              const float4 gt = slot_sum(a[j], lg);
              float4 up;
              up.x = __shfl_down_sync(0xffffffffu, gt.x, 4);
              up.y = __shfl_down_sync(0xffffffffu, gt.y, 4);
              up.z = __shfl_down_sync(0xffffffffu, gt.z, 4);
              up.w = __shfl_down_sync(0xffffffffu, gt.w, 4);
              const int f = f0 + tid + j * NT;
              if (f < T4 && ((f >> 3) & ((1 << lg) - 1)) == 0 && (f & 7) < 4)
                put(((f >> (3 + lg)) << 2) + (f & 7),
                    make_float4(silu_fast(gt.x) * up.x, silu_fast(gt.y) * up.y, silu_fast(gt.z) * up.z,
                                silu_fast(gt.w) * up.w));
            }
          }
        } else if (P.in_mode == IN_ATTN && step_splits(spos + 1, sp.P, HD) <= kSDefer) {
          // o = merge of the attention splits: sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s
          const int P_eff = step_splits(spos + 1, sp.P, HD);
          for (int r0 = 0; r0 < n4; r0 += 2 * NT) {
            float4 o[2][kSDefer];
            float2 ml[2][kSDefer];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              const int i4 = r0 + q * NT + tid;
              const int h = (4 * i4) / HD, d = (4 * i4) % HD, g = h / GQ, hh = h % GQ;
#pragma unroll
              for (int s = 0; s < kSDefer; ++s) {
                const bool pr = i4 < n4 && s < P_eff;
                const size_t base = ((size_t)g * sp.P + s) * GQ + hh;
                o[q][s] = ldcg4_if(sp.attn_o + base * HD + d, pr);
                ml[q][s] = ldcg2_if(sp.attn_ml + base * 2, pr);
              }
            }
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              const int i4 = r0 + q * NT + tid;
              if (i4 < n4) {
                float M = ml[q][0].x;
#pragma unroll
                for (int s = 1; s < kSDefer; ++s)
                  if (s < P_eff) M = fmaxf(M, ml[q][s].x);
                float L = 0.f;
                float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int s = 0; s < kSDefer; ++s)
                  if (s < P_eff) {
                    const float f = exp2f(ml[q][s].x - M);
                    L += ml[q][s].y * f;
                    O.x += o[q][s].x * f;
                    O.y += o[q][s].y * f;
                    O.z += o[q][s].z * f;
                    O.w += o[q][s].w * f;
                  }
                const float il = 1.0f / L;
                put(i4, make_float4(O.x * il, O.y * il, O.z * il, O.w * il));
              }
            }
          }
        } else {
          // embedding row of the token, or a plain vector (the merged attention output)
          const bool emb = P.in_mode == IN_EMBED_F32 || P.in_mode == IN_EMBED_BF16;
          int t = 0;
          if (emb) {
            t = *sp.tok;
            if (t < 0 || t >= sp.vocab) {
              if (tid == 0) atomicOr(sp.status, ST_BAD_TOKEN);
              t = 0;
            }
          }
          const float* src = P.in_mode == IN_ATTN ? sp.obuf : P.in_base;
          float4 v[kSMaxV];
#pragma unroll
          for (int j = 0; j < kSMaxV; ++j) {
            const int i = tid + j * NT;
            if (P.in_mode == IN_EMBED_BF16) {
              v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
              if (i < n4) {
                const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(sp.embed) +
                                                                      (size_t)t * K) + i);
                v[j] = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                                   __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
              }
            } else if (P.in_mode == IN_EMBED_F32) {
              v[j] = ldnc4_if(static_cast<const float*>(sp.embed) + (size_t)t * K + 4 * i, i < n4);
            } else {
              v[j] = ldcg4_if(src + 4 * i, i < n4);
            }
          }
#pragma unroll
          for (int j = 0; j < kSMaxV; ++j)
            if (tid + j * NT < n4) {
              if (emb) xr4[tid + j * NT] = v[j];  // the residual stream starts at the embedding
              put(tid + j * NT, v[j]);
            }
        }
        // RMSNorm factor over the whole vector
        float inv = 1.f;
        if (P.norm_w) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
          if (lane == 0) sm.bred[warp] = ss;
        }
        ConsumerSync::sync();  // publishes xh (written in row order by other threads)
        if (P.norm_w) {
          float t = 0.f;
#pragma unroll
          for (int w = 0; w < kSWarps; ++w) t += sm.bred[w];
          inv = 1.0f / sqrtf(t / (float)K + sp.eps);
        }
        // normalise in place (x / rms * w); per-group sums for the 4-bit units
#pragma unroll
        for (int j = 0; j < kSMaxV; ++j) {
          const int i = tid + j * NT;
          if (j * NT >= n4) break;  // uniform
          float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
          if (i < n4) {
            x = xh4[i];
            if (P.norm_w) {
              const float4 w = w4[j];
              x = make_float4(x.x * inv * w.x, x.y * inv * w.y, x.z * inv * w.z, x.w * inv * w.w);
              xh4[i] = x;
            }
          }
          if (!P.bf16) {  // the 16 threads holding a group of 64 inputs
            float gs = (x.x + x.y) + (x.z + x.w);
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) gs += __shfl_xor_sync(0xffffffffu, gs, o);
            if (i < n4 && (lane & 15) == 0) sm.u.g.xs[i / 16] = gs;
          }
        }
        for (int i = tid; i < kSRLoc * kSWarps * 32; i += NT) (&sm.u.g.red[0][0][0])[i] = 0.f;
        if (tid < 2) sm.carry_rt[tid] = -1;
        ConsumerSync::sync();

        // ---------------- stream the units; chunk i = units u0+15i .. u0+15i+14
        const int G = P.G, EPU = P.bf16 ? kBF16UnitCols : 64;
        int win_first = 0, win_idx = 0, win_rt0 = rt0, cur_rt = -1;
        float acc = 0.f;
        bool ok = true;
        for (int i = 0; i < n_chunks; ++i, ++gi) {
          const int s = gi % kSNSlot;
          if (ok) {
            ok = ring_wait(&full[s], (gi / kSNSlot) & 1, sp);
            if (!ok) *(volatile int*)&sm.abort = 1;
          }
          const int k = u0 + i * kSChunk + warp;
          if (ok && k < u1) {
            if (k_rt != cur_rt) {
              if (cur_rt >= 0) sm.u.g.red[cur_rt - win_rt0][warp][lane] = acc;
              acc = 0.f;
              cur_rt = k_rt;
            }
            const uint8_t* ub = ring + s * kSSlot + warp * P.unit_bytes;
            if (P.bf16) acc += bf16_unit_dot(ub, sm.u.g.xh + k_g * EPU, lane);
            else acc += q4_unit_dot(ub, sm.u.g.xh + k_g * EPU, sm.u.g.xs[k_g], lane);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
          k_g += kSChunk;
          while (k_g >= G) {
            k_g -= G;
            ++k_rt;
          }
          if (i + 1 == n_chunks || i + 1 - win_first == wch) {
            // close the reduction window: warps in order; every finished row
            // tile leaves this CTA's slot, a tile running on is carried
            if (cur_rt >= 0) sm.u.g.red[cur_rt - win_rt0][warp][lane] = acc;
            acc = 0.f;
            cur_rt = -1;
            ConsumerSync::sync();
            const int wu0 = u0 + win_first * kSChunk;
            const int wu1 = min(u1, u0 + (i + 1) * kSChunk);
            const int rt_a = wu0 / G, rt_b = (wu1 - 1) / G;
            const int next_rt = (wu1 < u1) ? wu1 / G : -1;
            const int carry_in_rt = sm.carry_rt[(win_idx + 1) & 1];
            for (int r = rt_a + warp; r <= rt_b; r += kSWarps) {
              const int li = r - rt_a;
              float sum = (r == carry_in_rt) ? sm.u.g.carry[(win_idx + 1) & 1][lane] : 0.f;
#pragma unroll
              for (int w2 = 0; w2 < kSWarps; ++w2) {
                sum += sm.u.g.red[li][w2][lane];
                sm.u.g.red[li][w2][lane] = 0.f;
              }
              if (r == next_rt) sm.u.g.carry[win_idx & 1][lane] = sum;
              else P.out_part[((size_t)r * P.part.S + (c - P.part.first_cta(r))) * 32 + lane] = sum;
            }
            if (tid == 0) sm.carry_rt[win_idx & 1] = (next_rt == rt_b) ? rt_b : -1;
            ConsumerSync::sync();
            win_first = i + 1;
            win_rt0 = next_rt;
            ++win_idx;
          }
        }
        // every warp passed the last window's closing barrier: the flag is uniform
        if (*(volatile int*)&sm.abort) break;
      } else if (P.type == PH_ATTN) {
        // ---------------- attention items (kv head, split) over the CTAs
        const int pos = spos;
        if (pos < 0 || pos >= sp.cap) {
          if (tid == 0 && c == 0) atomicOr(sp.status, ST_CTX_FULL);
        } else {
          const int P_eff = step_splits(pos + 1, sp.P, HD);
          for (int item = c; item < sp.Hkv * P_eff; item += N) {
            step_attn_item<GQ, HD>(sp, P, item / P_eff, item % P_eff, P_eff, pos, sm.u.a);
            ConsumerSync::sync();  // shared memory is reused by the next item
          }
        }
      } else {
        // ---------------- logits = sum of LM-head partials; greedy choice
        const int V = P.vocab;
        const int r0 = (int)((int64_t)V * c / N), r1 = (int)((int64_t)V * (c + 1) / N);
        const int lS = P.lm_S;
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        bool nan = false;
        constexpr int RR = 4;  // rows per thread per round
        for (int rb = r0; rb < r1; rb += RR * NT) {
          float y[RR][4];
#pragma unroll
          for (int j = 0; j < RR; ++j) {
            const int r = rb + tid + j * NT;
            const float* src = P.lm_part + ((size_t)(r >> 5) * lS) * 32 + (r & 31);
#pragma unroll
            for (int s = 0; s < 4; ++s) y[j][s] = ldcg1_if(src + s * 32, r < r1 && s < lS);
          }
#pragma unroll
          for (int j = 0; j < RR; ++j) {
            const int r = rb + tid + j * NT;
            if (r < r1) {
              const float v = (y[j][0] + y[j][1]) + (y[j][2] + y[j][3]);
              sp.logits[r] = v;
              if (v != v) nan = true;
              else if (better(v, r, bv, bi)) { bv = v; bi = r; }
            }
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
          sm.u.l.fbest[warp] = bv;
          sm.u.l.ibest[warp] = bi;
        }
        ConsumerSync::sync();
        if (tid == 0) {
          for (int w = 0; w < kSWarps; ++w)
            if (better(sm.u.l.fbest[w], sm.u.l.ibest[w], bv, bi)) { bv = sm.u.l.fbest[w]; bi = sm.u.l.ibest[w]; }
          sp.cand_v[c] = bv;
          sp.cand_i[c] = bi;
          __threadfence();
          sm.u.l.last = atomicAdd(sp.gcounter, 1) == N - 1;
        }
        ConsumerSync::sync();
        if (sm.u.l.last) {
          __threadfence();
          bv = -INFINITY;
          bi = 0x7fffffff;
          for (int k = tid; k < N; k += NT) {
            const float v2 = __ldcg(sp.cand_v + k);
            const int i2 = __ldcg(sp.cand_i + k);
            if (better(v2, i2, bv, bi)) { bv = v2; bi = i2; }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
          }
          ConsumerSync::sync();
          if (lane == 0) {
            sm.u.l.fbest[warp] = bv;
            sm.u.l.ibest[warp] = bi;
          }
          ConsumerSync::sync();
          if (tid == 0) {
            for (int w = 0; w < kSWarps; ++w)
              if (better(sm.u.l.fbest[w], sm.u.l.ibest[w], bv, bi)) { bv = sm.u.l.fbest[w]; bi = sm.u.l.ibest[w]; }
            if (bi < 0 || bi >= V) bi = 0;  // every logit NaN (status already says so)
            *sp.argmax_out = bi;
            *sp.tok_io = bi;
            const int h = *sp.hist_ctr;
            if (h < sp.hist_cap) sp.hist[h] = bi;
            *sp.hist_ctr = h + 1;
            *sp.pos = *sp.pos + 1;
            *sp.gcounter = 0;
          }
        }
      }
      if (ph + 1 < sp.n_phases) grid_arrive(sp);  // its CTA barrier also retires this phase's reads of sm.ph
    }
  }
  __syncthreads();
  // After an abort, wait (bounded) for copies still landing in the ring.
  if (sm.abort && tid == kSWarps * 32) {
    const int issued = sm.issued;
    for (int i = max(0, issued - kSNSlot); i < issued; ++i) {
      const unsigned long long t0 = globaltimer();
      while (!mbar_try_wait(&full[i % kSNSlot], (i / kSNSlot) & 1) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
  }
}

template <int GQ, int HD>
constexpr size_t step_smem_bytes() {
  return kSRing + ((sizeof(StepSmem<GQ, HD>) + 15) & ~size_t(15)) + 2 * kSNSlot * sizeof(uint64_t);
}

}  // namespace llmq
