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
// Split-K by input ranges: the K inputs of every GEMV are cut into R equal
// ranges and the CTAs into R equal groups; a CTA of group r computes whole row
// tiles over range r only, so it gathers just that range of its input vector
// and every row tile ends with exactly one partial sum per range (R slots).
// The next phase adds the slots while it builds its input (residual add,
// SwiGLU, attention-split merge are fused there); no phase needs a fix-up of
// its own and no float atomics are used. RMSNorm is linear in the GEMV
// after the per-vector factor 1/rms, so a CTA multiplies its range by the
// norm weight only and publishes the range's sum of squares; whoever reads
// the GEMV's output adds the R sums and applies 1/rms there. Every input
// build issues all of its loads before it uses any of them: one L2 round trip
// per phase.
//
// Attention is flash-decoding over (kv head, split) items. An item requests
// its cached K/V rows (asynchronous copies into padded shared-memory tiles)
// before the grid barrier that its q|k|v wait for; each warp then scores all
// GQ heads against 16 positions on the tensor cores (attn_mma.cuh). In the
// split variant the items run in their own phase and leave an unnormalised
// partial (o, max, sum) per split; with few splits the o-projection's input
// build merges them, so the merge costs no round trip of its own, and with
// many splits (long caches) the last split of a kv head merges them. In the
// FUSED variant (short caches, one kv head per o-projection range) every CTA
// runs the one item of its range inside the o-projection's input build and
// the attention phase is skipped.
#pragma once
#include "kernels.cuh"
#include "attn_mma.cuh"

#ifndef LLMQ_PHASE_STAMPS
#define LLMQ_PHASE_STAMPS 0  // 1: per-phase clock stamps for llm_phase_times (a measurement build: they cost
                             // the fused kernel registers, ~14 us per TinyLlama-1.1B token)
#endif
#ifndef LLMQ_UNIT_STAMPS
#define LLMQ_UNIT_STAMPS 0  // 1: llm_phase_times also records per-warp unit wait / dot cycles (measurement build)
#endif
#ifndef LLMQ_ATTN_CUDA_CORES
#define LLMQ_ATTN_CUDA_CORES 0  // 1: the step's attention blocks on the CUDA cores (comparison build)
#endif

namespace llmq {

// 15 consumer warps + 1 producer warp = 4 warps per scheduler, 128 registers each
constexpr bool kUnitStamps = LLMQ_UNIT_STAMPS != 0;
constexpr int kSWarps = 15;                      // consumer warps
constexpr int kSCThreads = kSWarps * 32;         // consumer threads
constexpr int kSThreads = kSCThreads + 32;       // + one producer warp
constexpr int kSChunk = kSWarps;                 // units per ring slot: one per consumer warp
constexpr int kSSlot = kSChunk * kQ4UnitBytes;   // 17280 B (bf16 chunks use 15360 B)
constexpr int kSNSlot = 8;
constexpr int kSRing = kSNSlot * kSSlot;         // 138240 B
constexpr int kSRLoc = 14;                       // row tiles a reduction window may touch
constexpr int kSMaxV = (kMaxK / 4 + kSCThreads - 1) / kSCThreads;  // float4s of a K-vector per thread
constexpr int kSDefer = 4;                       // splits the o-projection's input build merges
constexpr int kSMaxDim = 4096;                   // widest residual stream (kept in shared memory)
constexpr int kSFuseOut = 1024;                  // attention outputs a CTA computes for its o-projection range
constexpr int kSMaxW = (kSMaxDim / 4 + kSCThreads - 1) / kSCThreads;  // float4s of a norm weight per thread

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
  const uint8_t* units;   // [n_rt][G] units
  int n_rt, G, K, bf16, unit_bytes;
  int GR;                 // groups (units) of a row tile per input range: G / R
  float* out_part;        // [n_rt][R][32]: slot r = the sum over input range r
  int in_mode;
  const float* in_base;   // IN_PLAIN: the vector
  const float* in_part;   // IN_RESID / IN_SWIGLU: partials of the previous GEMV ([tile][R][32])
  float* in_store;        // the first CTA of each range stores its range of the built (pre-norm) vector, or null
  const float* norm_w;    // RMSNorm weight, or null
  float* ss_out;          // [4]: sum of squares of the pre-norm input over range r (norm phases)
  const float* ss_in;     // [4]: the sums of the GEMV whose output this phase reads (null: no norm)
  // ---- ATTN
  const float* qkv_part;
  const float* q_norm;
  const float* k_norm;
  // ---- LOGITS
  const float* lm_part;
  int vocab;
};

// The CTAs [floor(rN/R), floor((r+1)N/R)) serve input range r; CTA c of that
// group takes the row tiles [n_rt (c-c0) / nr, n_rt (c-c0+1) / nr).
struct KRange {
  int r, c0, nr;
  __host__ __device__ KRange(int c, int N, int R) {
    r = ((c + 1) * R - 1) / N;
    c0 = r * N / R;
    nr = (r + 1) * N / R - c0;
  }
  __host__ __device__ int tile(int c, int n_rt) const { return (int)((unsigned)n_rt * (unsigned)(c - c0) / (unsigned)nr); }
};

// 1/rms of a vector of `dim` elements from the per-range sums of squares
// (unused entries are zero), added in a fixed order.
__device__ __forceinline__ float rms_inv(float4 ss, int dim, float eps) {
  return 1.0f / sqrtf(((ss.x + ss.y) + (ss.z + ss.w)) / (float)dim + eps);
}

struct StepParams {
  const Phase* phases;
  int n_phases;
  int R;                  // input ranges of every GEMV (1, 2 or 4); slots per row tile
  int dim;                // residual width (RMSNorm mean)
  int* sync;              // [0] arrivals (phases x CTAs), [1] abort; zeroed before each launch
  int* status;
  int bar_extra;          // arrivals every grid barrier waits for beyond its CTAs (0; 1 in the expiry test)
  unsigned long long* stamps;  // measurement: [phase][CTA][16] clock64 stamps, or null
  unsigned long long wait_ns;  // limit of every wait on another CTA or on the ring
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
  int8_t* k8_base;        // the grouped int8 cache instead (int8 K/V models): codes [L][Hkv][cap][hd]
  int8_t* v8_base;
  uint16_t* ks_base;      // and fp16 scales of each 32-element group [L][Hkv][cap][hd / 32]
  uint16_t* vs_base;
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

// A wait's limit in SM cycles: the time limit at 2.1 cycles per ns (GB300's
// top clock; at lower clocks the limit only lasts longer).
__device__ __forceinline__ long long wait_cycles(const StepParams& sp) {
  return (long long)(sp.wait_ns * 21ull / 10ull);
}

// Consumer-side grid barrier: wait until `target` arrivals (bounded). Any
// timeout sets the shared abort flag, which ends every other wait at once.
__device__ inline bool grid_wait(const StepParams& sp, int target, int* s_flag) {
  target += sp.bar_extra;
  if (threadIdx.x == 0) {
    int ok = 1;
    if (ld_acquire(sp.sync) < target) {
      // polled without pauses (a pause only delays seeing the last arrival);
      // the abort word and the clock are read every 16th poll
      const long long c0 = clock64();
      for (unsigned it = 1; ld_acquire(sp.sync) < target; ++it) {
        if (it & 15) continue;
        if (*(volatile int*)(sp.sync + 1)) { ok = 0; break; }
        if (clock64() - c0 > wait_cycles(sp)) {
          atomicOr(sp.status, ST_TIMEOUT);
          atomicExch(sp.sync + 1, 1);
          ok = 0;
          break;
        }
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
  const long long c0 = clock64();
  for (unsigned it = 1; !mbar_try_wait(bar, parity); ++it) {
    if (it & 63) continue;  // the abort word and the clock every 64th try
    if (*(volatile int*)(sp.sync + 1)) return false;
    if (clock64() - c0 > wait_cycles(sp)) {
      atomicOr(sp.status, ST_TIMEOUT);
      atomicExch(sp.sync + 1, 1);
      return false;
    }
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
  __align__(16) uint16_t ksc[PP][HD / 32];  // int8 K/V: fp16 group scales of the staged rows
  __align__(16) uint16_t vsc[PP][HD / 32];
  float cursc[2][HD / 32];    // int8 K/V: this step's k, v group scales (cur then holds their codes)
  int is_last;
};

template <int GQ, int HD>
struct StepSmem {
  union {
    struct {
      float xh[kMaxK];                     // input vector of the GEMV (4-bit phases: its limbs, in place)
      float xs[kMaxK / 64];                // its per-group sums
      float fe[kMaxK / 64];                // 2^-sh / 16 of each group's fixed point
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
  __align__(16) float xres[kSMaxDim];  // this CTA's range of the residual stream (pre-norm)
  float fo[kSFuseOut];                 // attention output of this CTA's o-projection range
  Phase ph[2];            // descriptors of the current and the next phase
  int rt[2];              // this CTA's row tiles [rt[0], rt[1]) in the current GEMV phase
  float bred[kSWarps];
  int carry_rt[2];
  int flag;
  int abort;
  int issued;
};

// ---------------------------------------------------------------------------
// The first pass's K/V rows t0 .. of an attention item straight into its tiles
// (raw bf16, asynchronous copies). The cached rows were appended by earlier
// steps, so this runs before the grid barrier that the item's q|k|v wait for;
// row `pos` and the zero rows are written by the item. Thread-to-chunk map of
// step_attn_item's tile loads.
template <int GQ, int HD, bool KV8>
__device__ void step_attn_prefetch(const StepParams& sp, int layer, int g, int t0, int t1, int pos,
                                   StepAttnSmem<GQ, HD>& sa) {
  using SA = StepAttnSmem<GQ, HD>;
  constexpr int NT = kSCThreads, PP = SA::PP, CH = HD / 8;
  constexpr int TB = (2 * PP * CH + NT - 1) / NT;
  const int tid = threadIdx.x;
  if constexpr (KV8) {
    // one thread per staged row: its codes into the first HD bytes of the
    // row's fp16 slot (widened in place by the same thread), its scales beside
    static_assert(2 * PP <= NT, "one row per thread");
    constexpr int NG = HD / 32;
    const size_t cbase = (size_t)layer * sp.layer_stride + (size_t)g * sp.cap * HD;
    const int n = min(PP, t1 - t0);
    const int kv = tid / PP, row = tid - kv * PP;
    if (kv < 2 && row < n && t0 + row != pos && in_bounds(sp.status, t0 + row < sp.cap)) {
      const int8_t* src = (kv ? sp.v8_base : sp.k8_base) + cbase + (size_t)(t0 + row) * HD;
      uint8_t* dst = reinterpret_cast<uint8_t*>(&(kv ? sa.vt : sa.kt)[row][0]);
#pragma unroll
      for (int c = 0; c < HD / 16; ++c) cp_async16(dst + 16 * c, src + 16 * c);
      cp_async_small<2 * NG>(&(kv ? sa.vsc : sa.ksc)[row][0],
                             (kv ? sp.vs_base : sp.ks_base) + cbase / 32 + (size_t)(t0 + row) * NG);
    }
    return;
  }
  const uint16_t* kc = sp.k_base + (size_t)layer * sp.layer_stride + (size_t)g * sp.cap * HD;
  const uint16_t* vc = sp.v_base + (size_t)layer * sp.layer_stride + (size_t)g * sp.cap * HD;
  const int n = min(PP, t1 - t0);
#pragma unroll
  for (int j = 0; j < TB; ++j) {
    const int idx = tid + j * NT, kv = idx / (PP * CH), rem = idx - kv * (PP * CH), row = rem / CH, ch = rem - row * CH;
    if (kv < 2 && row < n && t0 + row != pos && in_bounds(sp.status, t0 + row < sp.cap))
      cp_async16(&(kv ? sa.vt : sa.kt)[row][8 * ch], (kv ? vc : kc) + (size_t)(t0 + row) * HD + 8 * ch);
  }
}

// ---------------------------------------------------------------------------
// One (kv head g, split) attention item, run by the consumer warps. `append`:
// this item writes the step's k, v into the cache. With `fo` null the item
// leaves its split's unnormalised partial (o, max, sum) in global memory;
// otherwise (one split over the whole cache) it writes the normalised output
// of its GQ heads to fo[h * HD + d] in shared memory.
template <int GQ, int HD, bool KV8>
__device__ void step_attn_item(const StepParams& sp, const Phase& P, int g, int split, int P_eff, int pos,
                               StepAttnSmem<GQ, HD>& sa, bool append, float* fo, bool prefetched) {
  using SA = StepAttnSmem<GQ, HD>;
  constexpr int NT = kSCThreads, PP = SA::PP, RS = SA::RS, CH = HD / 8;
  constexpr int TB = (2 * PP * CH + NT - 1) / NT;  // 16-B tile loads per thread
  static_assert((GQ + 1) * (HD / 2) + HD <= NT && GQ <= 8 && SA::NBW <= kSWarps,
                "one RoPE pair or v element per thread, GQ <= 8");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int len = pos + 1;
  const int t0 = (int)((int64_t)len * split / P_eff), t1 = (int)((int64_t)len * (split + 1) / P_eff);
  constexpr int NG = HD / 32;
  const size_t cbase = (size_t)P.layer * sp.layer_stride + (size_t)g * sp.cap * HD;
  uint16_t* kc = KV8 ? nullptr : sp.k_base + cbase;
  uint16_t* vc = KV8 ? nullptr : sp.v_base + cbase;
  int8_t* kc8 = KV8 ? sp.k8_base + cbase : nullptr;  // int8 K/V: codes and group scales
  int8_t* vc8 = KV8 ? sp.v8_base + cbase : nullptr;
  uint16_t* ks8 = KV8 ? sp.ks_base + cbase / 32 : nullptr;
  uint16_t* vs8 = KV8 ? sp.vs_base + cbase / 32 : nullptr;
  // int8 K/V: a row's HD codes (in registers) as fp16 halves (exact) into its tile row
  auto write_row_f16 = [&](uint16_t* tr, const uint4 (&c)[HD / 16]) {
#pragma unroll
    for (int k = HD / 16 - 1; k >= 0; --k) {  // from the end: the codes may sit in the row's first bytes
      const uint32_t w[4] = {c[k].x, c[k].y, c[k].z, c[k].w};
      uint32_t h[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float b0 = (float)(int8_t)(w[q] & 0xFF), b1 = (float)(int8_t)((w[q] >> 8) & 0xFF);
        const float b2 = (float)(int8_t)((w[q] >> 16) & 0xFF), b3 = (float)(int8_t)(w[q] >> 24);
        h[2 * q] = pack_f16x2(b0, b1);
        h[2 * q + 1] = pack_f16x2(b2, b3);
      }
      reinterpret_cast<uint4*>(tr)[2 * k] = make_uint4(h[0], h[1], h[2], h[3]);
      reinterpret_cast<uint4*>(tr)[2 * k + 1] = make_uint4(h[4], h[5], h[6], h[7]);
    }
  };
  // int8 K/V, the first pass: one thread per staged row widens the codes its
  // own asynchronous copies left in the first HD bytes of the row's slot, and
  // zero-fills rows n .. `rows` (codes and scales); row `pos` is left to this
  // step's k, v
  auto widen_rows = [&](int n, int rows) {
    const int kv = tid / PP, row = tid - kv * PP;
    if (kv < 2 && row < rows && t0 + row != pos) {
      uint16_t* tr = &(kv ? sa.vt : sa.kt)[row][0];
      uint4 c[HD / 16];
#pragma unroll
      for (int k = 0; k < HD / 16; ++k)
        c[k] = row < n ? reinterpret_cast<const uint4*>(tr)[k] : make_uint4(0u, 0u, 0u, 0u);
      write_row_f16(tr, c);
      if (row >= n)
#pragma unroll
        for (int k = 0; k < NG; ++k) (kv ? sa.vsc : sa.ksc)[row][k] = 0;
    }
  };

  // K/V rows tp .. tp+n-1 -> registers (zero beyond the split); stored into
  // the padded tiles once the previous readers are done. Row `pos` is left to
  // this step's k, v (another CTA may be appending it to the cache meanwhile).
  uint4 tl[KV8 ? HD / 16 : TB];
  uint2 tsc = make_uint2(0u, 0u);  // int8 K/V: the row's group scales (NG halves)
  auto load_tile = [&](int tp) {
    if constexpr (KV8) {
      const int n = min(PP, t1 - tp);
      const int kv = tid / PP, row = tid - kv * PP;
      const bool ld = kv < 2 && row < n && tp + row != pos && in_bounds(sp.status, tp + row < sp.cap);
      const int8_t* src = (kv ? vc8 : kc8) + (size_t)(tp + row) * HD;
#pragma unroll
      for (int k = 0; k < HD / 16; ++k) {
        const float4 v = ldcg4_if(reinterpret_cast<const float*>(src + 16 * k), ld);
        tl[k] = make_uint4(__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z), __float_as_uint(v.w));
      }
      const uint16_t* ssrc = (kv ? vs8 : ks8) + (size_t)(tp + row) * NG;
      if (ld) {
        if constexpr (NG == 2) tsc.x = __ldcg(reinterpret_cast<const unsigned int*>(ssrc));
        else tsc = __ldcg(reinterpret_cast<const uint2*>(ssrc));
      }
      return;
    }
    const int n = min(PP, t1 - tp);
#pragma unroll
    for (int j = 0; j < TB; ++j) {
      const int idx = tid + j * NT, kv = idx / (PP * CH), rem = idx - kv * (PP * CH), row = rem / CH, ch = rem - row * CH;
      const float4 v = ldcg4_if(reinterpret_cast<const float*>((kv ? vc : kc) + (size_t)(tp + row) * HD + 8 * ch),
                                kv < 2 && row < n && tp + row != pos && in_bounds(sp.status, tp + row < sp.cap));
      tl[j] = make_uint4(__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z), __float_as_uint(v.w));
    }
  };
  auto store_tile = [&](int tp) {
    if constexpr (KV8) {
      const int n = min(PP, t1 - tp), rows = ((n + 15) / 16) * 16;
      const int kv = tid / PP, row = tid - kv * PP;
      if (kv < 2 && row < rows && tp + row != pos) {
        if (row >= n)
#pragma unroll
          for (int k = 0; k < HD / 16; ++k) tl[k] = make_uint4(0u, 0u, 0u, 0u);
        write_row_f16(&(kv ? sa.vt : sa.kt)[row][0], tl);
        uint16_t* sc = &(kv ? sa.vsc : sa.ksc)[row][0];
        if constexpr (NG == 2) *reinterpret_cast<unsigned int*>(sc) = row < n ? tsc.x : 0u;
        else *reinterpret_cast<uint2*>(sc) = row < n ? tsc : make_uint2(0u, 0u);
      }
      return;
    }
    const int rows = ((min(PP, t1 - tp) + 15) / 16) * 16;
#pragma unroll
    for (int j = 0; j < TB; ++j) {
      const int idx = tid + j * NT, kv = idx / (PP * CH), rem = idx - kv * (PP * CH), row = rem / CH, ch = rem - row * CH;
      if (kv < 2 && row < rows && tp + row != pos)
        *reinterpret_cast<uint4*>(&(kv ? sa.vt : sa.kt)[row][8 * ch]) =
            make_uint4(bf16x2_to_f16x2(tl[j].x), bf16x2_to_f16x2(tl[j].y), bf16x2_to_f16x2(tl[j].z),
                       bf16x2_to_f16x2(tl[j].w));
    }
  };
  if (!prefetched) step_attn_prefetch<GQ, HD, KV8>(sp, P.layer, g, t0, t1, pos, sa);

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

  // ---- gather q (GQ heads), k and v of this kv head from the QKV partials;
  // the attention norm's 1/rms multiplies their sum
  {
    const float4 ssv = ldcg4_if(P.ss_in, true);
    const int lg = log2_slots(sp.R);
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
    const float inv = rms_inv(ssv, sp.dim, sp.eps);
#pragma unroll
    for (int j = 0; j < RB; ++j) {
      const float4 v = slot_sum(a[j], lg);
      const int f = tid + j * NT;
      if (f < T4 && ((f >> 3) & ((1 << lg) - 1)) == 0)
        *reinterpret_cast<float4*>(&sa.cur[0][0] + (f >> (3 + lg)) * 32 + (f & 7) * 4) =
            make_float4(v.x * inv, v.y * inv, v.z * inv, v.w * inv);
    }
  }
  {
    // the first pass's rows arrive by step_attn_prefetch: bf16 -> fp16 in place
    // (each thread its own chunks), zero rows up to the next multiple of 16
    cp_async_wait_all();
    const int n = min(PP, t1 - t0), rows = ((n + 15) / 16) * 16;
    if constexpr (KV8) widen_rows(n, rows);
#pragma unroll
    for (int j = 0; j < (KV8 ? 0 : TB); ++j) {
      const int idx = tid + j * NT, kv = idx / (PP * CH), rem = idx - kv * (PP * CH), row = rem / CH, ch = rem - row * CH;
      if (kv < 2 && row < rows && t0 + row != pos) {
        uint4* q = reinterpret_cast<uint4*>(&(kv ? sa.vt : sa.kt)[row][8 * ch]);
        const uint4 w = row < n ? *q : make_uint4(0u, 0u, 0u, 0u);
        *q = make_uint4(bf16x2_to_f16x2(w.x), bf16x2_to_f16x2(w.y), bf16x2_to_f16x2(w.z), bf16x2_to_f16x2(w.w));
      }
    }
  }
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
  const bool owner = t1 == len && pos - t0 < PP;  // the first pass's tile holds `pos`
  auto keep = [&](int r, int d, float x) {  // final value of cur[r][d], r >= GQ
    if constexpr (KV8) {  // quantized per 32-element group below
      sa.cur[r][d] = x;
      return;
    }
    const __nv_bfloat16 b = __float2bfloat16_rn(x);
    const float xr = __bfloat162float(b);
    sa.cur[r][d] = xr;
    if (append && in_bounds(sp.status, pos < sp.cap)) (r == GQ ? kc : vc)[(size_t)pos * HD + d] = __bfloat16_as_ushort(b);
    if (owner) (r == GQ ? sa.kt : sa.vt)[pos - t0][d] = __half_as_ushort(__float2half_rn(xr));
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
  if constexpr (KV8) {
    // the grouped int8 append: warp (kv, group) quantizes 32 elements of k or
    // v (fp16 scale fp16(amax / 127), codes round(x / scale) half away from
    // zero, clamped to +-127, all in fp32); cur keeps the codes, cursc the scales
    ConsumerSync::sync();
    if (warp < 2 * NG) {
      const int kv = warp / NG, grp = warp - kv * NG, d = 32 * grp + lane;
      const float x = sa.cur[GQ + kv][d];
      float amax = fabsf(x);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const __half dh = __float2half_rn(amax / 127.0f);
      const float dq = __half2float(dh);
      const float cf = dq == 0.0f ? 0.0f : fminf(fmaxf(roundf(x / dq), -127.0f), 127.0f);
      sa.cur[GQ + kv][d] = cf;
      if (lane == 0) sa.cursc[kv][grp] = dq;
      if (append && in_bounds(sp.status, pos < sp.cap)) {
        (kv ? vc8 : kc8)[(size_t)pos * HD + d] = (int8_t)(int)cf;
        if (lane == 0) (kv ? vs8 : ks8)[(size_t)pos * NG + grp] = __half_as_ushort(dh);
      }
      if (owner) {
        (kv ? sa.vt : sa.kt)[pos - t0][d] = __half_as_ushort(__float2half_rn(cf));
        if (lane == 0) (kv ? sa.vsc : sa.ksc)[pos - t0][grp] = __half_as_ushort(dh);
      }
    }
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
      if (pos >= tp && pos < tp + n) {
        for (int d = tid; d < HD; d += NT) {
          sa.kt[pos - tp][d] = __half_as_ushort(__float2half_rn(sa.cur[GQ][d]));
          sa.vt[pos - tp][d] = __half_as_ushort(__float2half_rn(sa.cur[GQ + 1][d]));
        }
        if constexpr (KV8)
          if (tid < 2 * NG)
            (tid < NG ? sa.ksc : sa.vsc)[pos - tp][tid % NG] =
                __half_as_ushort(__float2half_rn(sa.cursc[tid / NG][tid % NG]));
      }
      ConsumerSync::sync();
    }
    if (warp < nb) {
      if constexpr (KV8)
        attn_block16_q8<GQ, HD, RS>(&sa.cur[0][0], &sa.kt[0][0], &sa.vt[0][0], &sa.ksc[0][0], &sa.vsc[0][0],
                                    16 * warp, n - 16 * warp, lane, &sa.tres[warp][0][0], HD + 2);
      else
#if LLMQ_ATTN_CUDA_CORES
        attn_block16_cc<GQ, HD, RS>(&sa.cur[0][0], &sa.kt[0][0], &sa.vt[0][0], 16 * warp, n - 16 * warp, lane,
                                    &sa.tres[warp][0][0], HD + 2);
#else
        attn_block16<GQ, HD, RS>(&sa.cur[0][0], &sa.kt[0][0], &sa.vt[0][0], 16 * warp, n - 16 * warp, lane,
                                 &sa.tres[warp][0][0], HD + 2);
#endif
    }
    ConsumerSync::sync();
    // fold the pass into the running output. Warp h < GQ finds head h's
    // factors, lane w < nb for block w: new max, 2^(m_w - M), sum update
    if (warp < GQ) {
      const int h = warp;
      const float am = sa.accm[h], al = sa.accl[h];
      const float mw = lane < nb ? sa.tres[lane][h][HD] : -INFINITY;
      const float lw = lane < nb ? sa.tres[lane][h][HD + 1] : 0.f;
      float M = fmaxf(mw, am);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      const float f = lane < nb ? exp2f(mw - M) : 0.f;
      float L = lw * f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
      const float fa = am == -INFINITY ? 0.f : exp2f(am - M);
      __syncwarp();
      if (lane < SA::NBW) sa.fac[h][1 + lane] = f;
      if (lane == 0) {
        sa.fac[h][0] = fa;
        sa.accm[h] = M;
        sa.accl[h] = al * fa + L;
      }
    }
    ConsumerSync::sync();
    for (int i = tid; i < GQ * HD; i += NT) {
      const int h = i / HD, d = i % HD;
      float O = sa.acc[h][d] * sa.fac[h][0];
#pragma unroll
      for (int w = 0; w < SA::NBW; ++w)
        if (w < nb) O += sa.tres[w][h][d] * sa.fac[h][1 + w];
      sa.acc[h][d] = O;
    }
    // the next pass writes its tiles and blocks after the barrier of its staging
  }

  // ---- the output: every thread reads back the elements it folded
  if (fo) {
    for (int i = tid; i < GQ * HD; i += NT) fo[i] = sa.acc[i / HD][i % HD] / sa.accl[i / HD];
    return;
  }
  {
    const size_t pbase = ((size_t)g * sp.P + split) * GQ;
    for (int i = tid; i < GQ * HD; i += NT) {
      const int h = i / HD, d = i % HD;
      sp.attn_o[pbase * HD + i] = sa.acc[h][d];
      if (d == 0) {
        sp.attn_ml[(pbase + h) * 2] = sa.accm[h];
        sp.attn_ml[(pbase + h) * 2 + 1] = sa.accl[h];
      }
    }
  }

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

// FUSED: the variant for short caches (every CTA computes the attention of
// its o-projection range in that GEMV's input build; no attention phase). The
// two variants are separate kernels: either one alone keeps its registers.
template <int GQ, int HD, bool FUSED, bool A8, bool KV8>
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

  const KRange kr(c, N, sp.R);  // this CTA's input range in every GEMV phase
  if (LLMQ_PHASE_STAMPS && sp.stamps && tid == 0) {  // (%globaltimer, clock64) pairs map this SM's cycles onto one time line
    sp.stamps[(size_t)c * 16 + 12] = globaltimer();
    sp.stamps[(size_t)c * 16 + 13] = clock64();
  }
  if (warp == kSWarps) {
    // ================= producer: every GEMV phase's units, in phase order
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int gi = 0;
      bool ok = true;
      for (int ph = 0; ph < sp.n_phases && ok; ++ph) {
        const Phase& P = sp.phases[ph];
        if (P.type != PH_GEMV) continue;
        // this CTA's units in range order: v = tile * GR + (group - r * GR)
        const int GR = P.GR, UB = P.unit_bytes;
        const int u0 = kr.tile(c, P.n_rt) * GR, u1 = kr.tile(c + 1, P.n_rt) * GR;
        for (int ub = u0; ub < u1; ub += kSChunk, ++gi) {
          const int s = gi % kSNSlot;
          if (gi >= kSNSlot && !ring_wait(&empty[s], ((gi / kSNSlot) - 1) & 1, sp)) {
            ok = false;
            break;
          }
          const int ue = min(u1, ub + kSChunk);
          mbar_expect_tx(&full[s], (ue - ub) * UB);
          // one copy per row tile touched: the range's units of a tile are contiguous
          for (int v = ub; v < ue;) {
            const int rt = v / GR, gp = v - rt * GR, run = min(ue - v, GR - gp);
            // (checked build: an index outside the stream copies its first units instead, so
            // the slot still completes; the status word reports the error)
            const bool okc = in_bounds(sp.status, rt < P.n_rt && kr.r * GR + gp + run <= P.G &&
                                                      (v - ub + run) * UB <= kSSlot);
            bulk_g2s(ring + s * kSSlot + (v - ub) * UB,
                     P.units + (okc ? ((size_t)rt * P.G + kr.r * GR + gp) * UB : 0), run * UB, &full[s], pol);
            v += run;
          }
          sm.issued = gi + 1;
        }
      }
    }
  } else {
    // ================= consumers
    constexpr int NT = kSCThreads;
    constexpr bool a8 = A8;
    uint32_t mlo, mhi;  // the nibble masks of the unit dot, held in registers
    asm volatile("mov.b32 %0, 0x0F0F0F0F;" : "=r"(mlo));
    asm volatile("mov.b32 %0, 0xF0F0F0F0;" : "=r"(mhi));
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
    // the window sums are zero after a GEMV phase (every window close clears
    // what it read); attention and logit phases reuse their shared memory
    bool red_clear = false;
    // short caches: every CTA computes the attention of its o-projection range
    // while it builds that GEMV's input, and the attention phase is skipped
    constexpr bool fuse = FUSED;
    int bars = 0;  // grid barriers this CTA arrived at
    for (int ph = 0; ph < sp.n_phases; ++ph) {
      const Phase& P = sm.ph[ph & 1];
      // measurement stamps (tid 0): 0 phase start, 1 barrier passed, 2 input
      // built, 3 units done, 4 arrival issued
      unsigned long long* st =
          (LLMQ_PHASE_STAMPS && sp.stamps) ? sp.stamps + ((size_t)ph * N + c) * 16 : nullptr;
      if (st && tid == 0) st[0] = clock64();
      if (P.type == PH_ATTN && fuse) {
        fetch_phase(ph + 1);
        ConsumerSync::sync();
        red_clear = false;  // the o-projection's build reuses that shared memory
        continue;
      }
      const int Kr = P.type == PH_GEMV ? P.K / sp.R : 0;  // inputs of this CTA's range
      // norm weights do not depend on the step: in flight while the barrier resolves
      float4 w4[kSMaxW];
      {
        const bool nw = P.type == PH_GEMV && P.norm_w != nullptr;
#pragma unroll
        for (int j = 0; j < kSMaxW; ++j) {
          const int i = tid + j * NT;
          w4[j] = ldnc4_if(nw ? P.norm_w + kr.r * Kr + 4 * i : nullptr, nw && i < Kr / 4);
        }
      }
      // the units of this CTA in range order, v = tile * GR + group within the
      // range (divisions: done while the barrier resolves)
      // (kept in shared memory until the chunk loop: no registers held over the build)
      if (P.type == PH_GEMV && tid == 0) {
        sm.rt[0] = kr.tile(c, P.n_rt);
        sm.rt[1] = kr.tile(c + 1, P.n_rt);
      }
      // the next descriptor goes to the buffer the previous phase used: its
      // round trip overlaps the barrier wait
      fetch_phase(ph + 1);
      // attention: the cached K/V rows of this CTA's first item start arriving
      // while the barrier resolves (the union's previous user finished before
      // its phase's arrival)
      bool pf = false;
      if (spos >= 0 && spos < sp.cap) {
        if constexpr (FUSED) {
          if (P.type == PH_GEMV && P.in_mode == IN_ATTN) {
            step_attn_prefetch<GQ, HD, KV8>(sp, P.layer, kr.r * (sp.Hkv / sp.R), 0, spos + 1, spos, sm.u.a);
            pf = true;
          }
        } else if (P.type == PH_ATTN) {
          const int P_eff = step_splits(spos + 1, sp.P, HD);
          if (c < sp.Hkv * P_eff) {
            const int split = c % P_eff, len = spos + 1;
            const int t0 = (int)((int64_t)len * split / P_eff), t1 = (int)((int64_t)len * (split + 1) / P_eff);
            step_attn_prefetch<GQ, HD, KV8>(sp, P.layer, c / P_eff, t0, t1, spos, sm.u.a);
            pf = true;
          }
        }
      }
      if (ph > 0 && !grid_wait(sp, bars * N, &sm.flag)) {
        cp_async_wait_all();  // no copy may land after the CTA leaves
        sm.abort = 1;
        break;
      }
      if (st && tid == 0) st[1] = clock64();
      if (P.type == PH_GEMV) {
        // ---------------- build this CTA's range of the input vector (inputs
        // r*K .. r*K+K-1 of the GEMV): every load of the build in one round trip
        const int K = Kr, n4 = K / 4;
        const bool first = c == kr.c0;  // the range's first CTA publishes what all of its CTAs build
        float4* xh4 = reinterpret_cast<float4*>(sm.u.g.xh);
        float ss = 0.f;
        float4* xr4 = reinterpret_cast<float4*>(sm.xres);
        auto put = [&](int i4, float4 v) {  // pre-norm inputs r*K + 4*i4 .. +3
          xh4[i4] = v;
          if (P.in_store && first) reinterpret_cast<float4*>(P.in_store + kr.r * K)[i4] = v;
          ss += (v.x * v.x + v.y * v.y) + (v.z * v.z + v.w * v.w);
        };
        if (P.in_mode == IN_RESID) {
          // x = residual (this CTA's resident copy of its range) + sum of the
          // previous GEMV's slots (row tiles of 32 inputs); x becomes the new residual
          constexpr int RB = 8;
          const int lg = log2_slots(sp.R);
          const int T4 = (K / 32) << (3 + lg);
          const float* src = P.in_part + (size_t)kr.r * (K / 32) * (32 << lg);
          for (int f0 = 0; f0 < T4; f0 += RB * NT) {
            float4 a[RB];
#pragma unroll
            for (int j = 0; j < RB; ++j) {
              const int f = f0 + tid + j * NT;
              a[j] = ldcg4_if(src + (size_t)f * 4, f < T4);
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
          // row tile t of the gate|up GEMV: 16 gate rows, then their 16 up rows
          // -> inputs 16t..16t+15; both carry the FFN norm's 1/rms
          constexpr int RB = 12;
          const int lg = log2_slots(sp.R);
          const int T4 = (K / 16) << (3 + lg);
          const float* src = P.in_part + (size_t)kr.r * (K / 16) * (32 << lg);
          const float4 ssv = ldcg4_if(P.ss_in, true);
          for (int f0 = 0; f0 < T4; f0 += RB * NT) {
            float4 a[RB];
#pragma unroll
            for (int j = 0; j < RB; ++j) {
              const int f = f0 + tid + j * NT;
              a[j] = ldcg4_if(src + (size_t)f * 4, f < T4);
            }
            const float inv = rms_inv(ssv, sp.dim, sp.eps);
#pragma unroll
            for (int j = 0; j < RB; ++j) {
              float4 gt = slot_sum(a[j], lg);
              gt = make_float4(gt.x * inv, gt.y * inv, gt.z * inv, gt.w * inv);
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
        } else if (P.in_mode == IN_ATTN && fuse) {
          // the attention of the range's kv heads over the whole cache, here
          // (the range's first CTA appends k, v to the cache)
          const bool pos_ok = spos >= 0 && spos < sp.cap;  // else: the status says so, the step runs on zeros
          if (!pos_ok && tid == 0 && c == 0) atomicOr(sp.status, ST_CTX_FULL);
          const int hpr = sp.Hkv / sp.R;
          for (int j = 0; j < hpr && pos_ok; ++j) {
            step_attn_item<GQ, HD, KV8>(sp, P, kr.r * hpr + j, 0, 1, spos, sm.u.a, first, sm.fo + j * GQ * HD,
                                   j == 0 && pf);
            ConsumerSync::sync();  // the next item and the input vector reuse the shared memory
          }
          for (int i = tid; i < K; i += NT) sm.u.g.xh[i] = pos_ok ? sm.fo[i] : 0.f;
        } else if (P.in_mode == IN_ATTN && step_splits(spos + 1, sp.P, HD) <= kSDefer) {
          // o = merge of the attention splits: sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s
          const int P_eff = step_splits(spos + 1, sp.P, HD);
          for (int r0 = 0; r0 < n4; r0 += 2 * NT) {
            float4 o[2][kSDefer];
            float2 ml[2][kSDefer];
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              const int i4 = r0 + q * NT + tid, e = kr.r * K + 4 * i4;  // q_dim element
              const int h = e / HD, d = e % HD, g = h / GQ, hh = h % GQ;
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
          const float* src = (P.in_mode == IN_ATTN ? sp.obuf : P.in_base) + kr.r * K;
          float4 v[kSMaxV];
#pragma unroll
          for (int j = 0; j < kSMaxV; ++j) {
            const int i = tid + j * NT;
            if (P.in_mode == IN_EMBED_BF16) {
              v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
              if (i < n4) {
                const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(sp.embed) +
                                                                      (size_t)t * P.K + kr.r * K) + i);
                v[j] = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                                   __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
              }
            } else if (P.in_mode == IN_EMBED_F32) {
              v[j] = ldnc4_if(static_cast<const float*>(sp.embed) + (size_t)t * P.K + kr.r * K + 4 * i, i < n4);
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
        // the range's sum of squares (the readers of this GEMV apply 1/rms)
        if (P.norm_w) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
          if (lane == 0) sm.bred[warp] = ss;
        }
        ConsumerSync::sync();  // publishes xh (written in row order by other threads)
        if (P.norm_w && first && tid == 0) {
          float t = 0.f;
#pragma unroll
          for (int w = 0; w < kSWarps; ++w) t += sm.bred[w];
          P.ss_out[kr.r] = t;
        }
        // x * w (RMSNorm without its 1/rms), then what the units read: the
        // fp32 vector (bf16 units) or each group's limbs, exponent and sum
        // (4-bit units, in place of the group's floats)
#pragma unroll
        for (int j = 0; j < kSMaxV; ++j) {
          const int i = tid + j * NT;
          if (j * NT >= n4) break;  // uniform
          float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
          if (i < n4) {
            x = xh4[i];
            if (P.norm_w && j < kSMaxW) {  // normed inputs are residual-wide
              const float4 w = w4[j];
              x = make_float4(x.x * w.x, x.y * w.y, x.z * w.z, x.w * w.w);
            }
          }
          if (A8 && !P.bf16)
            q8_build_group(x, i, i < n4, sm.u.g.xh);
          else
            q4_build_group(x, i, i < n4, P.bf16 != 0, reinterpret_cast<uint4*>(sm.u.g.xh), sm.u.g.xh, sm.u.g.fe,
                           sm.u.g.xs);
        }
        if (!red_clear)
          for (int i = tid; i < kSRLoc * kSWarps * 32; i += NT) (&sm.u.g.red[0][0][0])[i] = 0.f;
        if (tid < 2) sm.carry_rt[tid] = -1;
        ConsumerSync::sync();
        if (st && tid == 0) st[2] = clock64();

        // ---------------- stream the units; chunk i = units u0+15i .. u0+15i+14
        const int G = P.GR, EPU = P.bf16 ? kBF16UnitCols : 64;
        const int rt0 = sm.rt[0], u0 = rt0 * G, u1 = sm.rt[1] * G;
        const int n_chunks = (u1 - u0 + kSChunk - 1) / kSChunk;
        const int wch = max(1, ((kSRLoc - 2) * G + 1) / kSChunk);
        int k_rt = rt0, k_g = warp;  // this warp's first unit: u0 + warp
        while (k_g >= G) {
          k_g -= G;
          ++k_rt;
        }
        int win_first = 0, win_idx = 0, win_rt0 = rt0, cur_rt = -1;
        float acc = 0.f;
        bool ok = true;
        long long t_wait = 0, t_dot = 0;  // measurement build (LLMQ_UNIT_STAMPS): cycles waiting / in unit dots
        for (int i = 0; i < n_chunks; ++i, ++gi) {
          const int s = gi % kSNSlot;
          const long long ta = (kUnitStamps && st) ? clock64() : 0;
          if (ok) {
            ok = ring_wait(&full[s], (gi / kSNSlot) & 1, sp);
            if (!ok) *(volatile int*)&sm.abort = 1;
          }
          const long long tb = (kUnitStamps && st) ? clock64() : 0;
          const int k = u0 + i * kSChunk + warp;
          if (ok && k < u1) {
            if (k_rt != cur_rt) {
              if (cur_rt >= 0) sm.u.g.red[cur_rt - win_rt0][warp][lane] = acc;
              acc = 0.f;
              cur_rt = k_rt;
            }
            const uint8_t* ub = ring + s * kSSlot + warp * P.unit_bytes;
            if (P.bf16) acc += bf16_unit_dot(ub, sm.u.g.xh + k_g * EPU, lane);
            else if (a8) acc += q4a8_unit_dot(ub, sm.u.g.xh + 64 * k_g, lane, mlo, mhi);
            else
              acc += q4_unit_dot_limbs(ub, reinterpret_cast<const uint4*>(sm.u.g.xh) + 16 * k_g, sm.u.g.fe[k_g],
                                       sm.u.g.xs[k_g], lane, mlo, mhi);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
          if (kUnitStamps && st) {
            t_wait += tb - ta;
            t_dot += clock64() - tb;
          }
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
            for (int t = rt_a + warp; t <= rt_b; t += kSWarps) {
              const int li = t - rt_a;
              float sum = (t == carry_in_rt) ? sm.u.g.carry[(win_idx + 1) & 1][lane] : 0.f;
#pragma unroll
              for (int w2 = 0; w2 < kSWarps; ++w2) {
                sum += sm.u.g.red[li][w2][lane];
                sm.u.g.red[li][w2][lane] = 0.f;
              }
              if (t == next_rt) sm.u.g.carry[win_idx & 1][lane] = sum;
              else if (in_bounds(sp.status, t < P.n_rt)) P.out_part[((size_t)t * sp.R + kr.r) * 32 + lane] = sum;
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
        if (kUnitStamps && st) {
          if (lane == 0) {
            sm.u.g.red[0][warp][0] = (float)t_wait;  // (the windows are closed: red is free)
            sm.u.g.red[0][warp][1] = (float)t_dot;
          }
          ConsumerSync::sync();
          if (tid == 0) {
            float mw = 0.f, md = 0.f, sw = 0.f, sd = 0.f;
            for (int w = 0; w < kSWarps; ++w) {
              mw = fmaxf(mw, sm.u.g.red[0][w][0]);
              md = fmaxf(md, sm.u.g.red[0][w][1]);
              sw += sm.u.g.red[0][w][0];
              sd += sm.u.g.red[0][w][1];
            }
            st[5] = (unsigned long long)mw;
            st[6] = (unsigned long long)md;
            st[7] = (unsigned long long)sw;
            st[8] = (unsigned long long)sd;
          }
          ConsumerSync::sync();
          if (lane == 0) {
            sm.u.g.red[0][warp][0] = 0.f;
            sm.u.g.red[0][warp][1] = 0.f;
          }
        }
        if (st && tid == 0) st[3] = clock64();
      } else if (P.type == PH_ATTN) {
        if constexpr (!FUSED) {
          // ---------------- attention items (kv head, split) over the CTAs
          const int pos = spos;
          if (pos < 0 || pos >= sp.cap) {
            if (tid == 0 && c == 0) atomicOr(sp.status, ST_CTX_FULL);
          } else {
            const int P_eff = step_splits(pos + 1, sp.P, HD);
            for (int item = c; item < sp.Hkv * P_eff; item += N) {
              step_attn_item<GQ, HD, KV8>(sp, P, item / P_eff, item % P_eff, P_eff, pos, sm.u.a,
                                     item % P_eff == P_eff - 1, nullptr, item == c && pf);
              ConsumerSync::sync();  // shared memory is reused by the next item
            }
          }
        }
      } else {
        // ---------------- logits = 1/rms (final norm) x sum of the LM-head
        // partials; greedy choice
        const int V = P.vocab;
        const int r0 = (int)((int64_t)V * c / N), r1 = (int)((int64_t)V * (c + 1) / N);
        const int lS = sp.R;
        const float4 ssv = ldcg4_if(P.ss_in, true);
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
          const float inv = rms_inv(ssv, sp.dim, sp.eps);
#pragma unroll
          for (int j = 0; j < RR; ++j) {
            const int r = rb + tid + j * NT;
            if (r < r1 && in_bounds(sp.status, r < V)) {
              const float v = ((y[j][0] + y[j][1]) + (y[j][2] + y[j][3])) * inv;
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
      red_clear = P.type == PH_GEMV;
      if (ph + 1 < sp.n_phases) {
        grid_arrive(sp);  // its CTA barrier also retires this phase's reads of sm.ph
        ++bars;
      }
      if (st && tid == 0) st[4] = clock64();
    }
  }
  __syncthreads();
  if (LLMQ_PHASE_STAMPS && sp.stamps && tid == 0) {
    sp.stamps[(size_t)c * 16 + 14] = globaltimer();
    sp.stamps[(size_t)c * 16 + 15] = clock64();
  }
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

// A kernel of a shape, as the host launches it: entry point and dynamic shared memory.
struct KernelRef {
  const void* fn = nullptr;
  size_t smem = 0;
};
// The step kernel for a GQA group, head_dim, variant, activation numerics and
// cache format (defined in step_kernels.cu and step_kernels_kv8.cu, which
// hold the instantiations); fn is null for an unsupported shape.
KernelRef step_kernel_ref(int gq, int hd, bool fused, bool w4a8, bool kv8);

}  // namespace llmq
