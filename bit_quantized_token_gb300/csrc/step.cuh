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
// Split-K across CTAs leaves one partial sum per CTA that touches a row tile;
// the next phase adds the slots in CTA order while it builds its input vector
// (residual add, SwiGLU, RMSNorm are fused there), so no phase needs a fix-up
// of its own and no float atomics are used.
#pragma once
#include "kernels.cuh"

namespace llmq {

// 15 consumer warps + 1 producer warp = 4 warps per scheduler, 128 registers each
constexpr int kSWarps = 15;                      // consumer warps
constexpr int kSThreads = (kSWarps + 1) * 32;    // + one producer warp
constexpr int kSChunk = kSWarps;                 // units per ring slot: one per consumer warp
constexpr int kSSlot = kSChunk * kQ4UnitBytes;   // 17280 B (bf16 chunks use 15360 B)
constexpr int kSNSlot = 8;
constexpr int kSRing = kSNSlot * kSSlot;         // 138240 B
constexpr int kSRLoc = 6;                        // row tiles a reduction window may touch

enum PhaseType : int { PH_GEMV = 0, PH_ATTN = 1, PH_LOGITS = 2 };
enum InMode : int { IN_EMBED_F32 = 0, IN_EMBED_BF16 = 1, IN_PLAIN = 2, IN_RESID = 3, IN_SWIGLU = 4 };

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
  int in_S;
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
  float* attn_part;
  int* attn_cnt;
  float* obuf;
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
  __device__ static void sync() { asm volatile("bar.sync 1, %0;" ::"n"(kSWarps * 32) : "memory"); }
};

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

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

// Bounded ring wait that also gives up when another CTA aborted the step.
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

// Sum of the S partial slots of 4 consecutive rows r..r+3 (same row tile).
__device__ __forceinline__ float4 reduce4(const float* __restrict__ part, int S, int r) {
  const float4* src = reinterpret_cast<const float4*>(part + ((size_t)(r >> 5) * S) * kTileRows + (r & 31));
  float4 a = __ldcg(src);
  for (int j = 1; j < S; ++j) {
    const float4 b = __ldcg(src + j * (kTileRows / 4));
    a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
  }
  return a;
}

template <int GQ, int HD>
struct StepSmem {
  union {
    struct {
      float xh[kMaxK];                     // input vector of the GEMV
      float xs[kMaxK / 64];                // its per-group sums
      float red[kSRLoc][kSWarps][32];      // per-warp row-tile sums of a window
      float carry[2][32];
    } g;
    AttnSmem<GQ, HD, kSWarps> a;
    struct {
      float fbest[kSWarps];
      int ibest[kSWarps];
      int last;
    } l;
  } u;
  Phase ph[2];            // descriptors of the current and the next phase
  float bred[kSWarps];
  int carry_rt[2];
  int flag;
  int abort;
  int issued;
};

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
    int gi = 0;
    // descriptors go to shared memory one phase ahead (the phase table is immutable)
    static_assert(sizeof(Phase) % 4 == 0, "");
    auto fetch_phase = [&](int ph) {
      if (ph < sp.n_phases)
        for (int i = tid; i < (int)(sizeof(Phase) / 4); i += kSWarps * 32)
          reinterpret_cast<int*>(&sm.ph[ph & 1])[i] = __ldg(reinterpret_cast<const int*>(&sp.phases[ph]) + i);
    };
    fetch_phase(0);
    ConsumerSync::sync();
    for (int ph = 0; ph < sp.n_phases; ++ph) {
      if (ph > 0 && !grid_wait(sp, ph * N, &sm.flag)) {
        sm.abort = 1;
        break;
      }
      const Phase& P = sm.ph[ph & 1];
      fetch_phase(ph + 1);  // read by the next phase, after this phase's closing barriers
      if (P.type == PH_GEMV) {
        // ---------------- build the input vector (thread t: float4s t, t+512, ...)
        constexpr int MAXV = (kMaxK / 4 + kSWarps * 32 - 1) / (kSWarps * 32);
        const int K = P.K, n4 = K / 4;
        float4 v[MAXV];
        if (P.in_mode == IN_EMBED_F32 || P.in_mode == IN_EMBED_BF16) {
          int t = *sp.tok;
          if (t < 0 || t >= sp.vocab) {
            if (tid == 0) atomicOr(sp.status, ST_BAD_TOKEN);
            t = 0;
          }
#pragma unroll
          for (int j = 0; j < MAXV; ++j) {
            const int i = tid + j * kSWarps * 32;
            if (i < n4) {
              if (P.in_mode == IN_EMBED_F32) {
                v[j] = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(sp.embed) + (size_t)t * K) + i);
              } else {
                const uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(sp.embed) + (size_t)t * K) + i);
                v[j] = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                                   __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
              }
            }
          }
        } else if (P.in_mode == IN_PLAIN) {
#pragma unroll
          for (int j = 0; j < MAXV; ++j) {
            const int i = tid + j * kSWarps * 32;
            if (i < n4) v[j] = __ldcg(reinterpret_cast<const float4*>(P.in_base) + i);
          }
        } else if (P.in_mode == IN_RESID) {
#pragma unroll
          for (int j = 0; j < MAXV; ++j) {
            const int i = tid + j * kSWarps * 32;
            if (i < n4) {
              const float4 b = __ldcg(reinterpret_cast<const float4*>(P.in_base) + i);
              const float4 a = reduce4(P.in_part, P.in_S, 4 * i);
              v[j] = make_float4(b.x + a.x, b.y + a.y, b.z + a.z, b.w + a.w);
            }
          }
        } else {  // IN_SWIGLU: gate rows 16t.., up rows 16t+16.. of row tile t
#pragma unroll
          for (int j = 0; j < MAXV; ++j) {
            const int i = tid + j * kSWarps * 32;
            if (i < n4) {
              const int e = 4 * i, r = (e >> 4) * 32 + (e & 15);
              const float4 gt = reduce4(P.in_part, P.in_S, r);
              const float4 up = reduce4(P.in_part, P.in_S, r + 16);
              v[j] = make_float4(silu_fast(gt.x) * up.x, silu_fast(gt.y) * up.y, silu_fast(gt.z) * up.z,
                                 silu_fast(gt.w) * up.w);
            }
          }
        }
        float4 nw4[MAXV];  // norm weights, loaded in the same round trip as the input
        if (P.norm_w)
#pragma unroll
          for (int j = 0; j < MAXV; ++j) {
            const int i = tid + j * kSWarps * 32;
            if (i < n4) nw4[j] = __ldg(reinterpret_cast<const float4*>(P.norm_w) + i);
          }
        if (P.in_store && c == 0)
#pragma unroll
          for (int j = 0; j < MAXV; ++j) {
            const int i = tid + j * kSWarps * 32;
            if (i < n4) reinterpret_cast<float4*>(P.in_store)[i] = v[j];
          }
        if (P.norm_w) {  // RMSNorm: x / sqrt(mean(x^2) + eps) * w
          float ss = 0.f;
#pragma unroll
          for (int j = 0; j < MAXV; ++j)
            if (tid + j * kSWarps * 32 < n4)
              ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
          if (lane == 0) sm.bred[warp] = ss;
          ConsumerSync::sync();
          ss = 0.f;
#pragma unroll
          for (int w = 0; w < kSWarps; ++w) ss += sm.bred[w];
          const float inv = 1.0f / sqrtf(ss / (float)K + sp.eps);
#pragma unroll
          for (int j = 0; j < MAXV; ++j) {
            const int i = tid + j * kSWarps * 32;
            if (i < n4) {
              const float4 w4 = nw4[j];
              v[j] = make_float4(v[j].x * inv * w4.x, v[j].y * inv * w4.y, v[j].z * inv * w4.z, v[j].w * inv * w4.w);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < MAXV; ++j) {
          const int i = tid + j * kSWarps * 32;
          if (j * kSWarps * 32 >= n4) break;  // uniform
          if (i < n4) reinterpret_cast<float4*>(sm.u.g.xh)[i] = v[j];
          if (!P.bf16) {  // per-group sums over the 16 threads holding a group
            float gs = (i < n4) ? (v[j].x + v[j].y) + (v[j].z + v[j].w) : 0.f;
#pragma unroll
            for (int o = 8; o > 0; o >>= 1) gs += __shfl_xor_sync(0xffffffffu, gs, o);
            if (i < n4 && (lane & 15) == 0) sm.u.g.xs[i / 16] = gs;
          }
        }
        for (int i = tid; i < kSRLoc * kSWarps * 32; i += kSWarps * 32) (&sm.u.g.red[0][0][0])[i] = 0.f;
        if (tid < 2) sm.carry_rt[tid] = -1;
        ConsumerSync::sync();

        // ---------------- stream the units; chunk i = units u0+16i .. u0+16i+15
        const int G = P.G, EPU = P.bf16 ? kBF16UnitCols : 64;
        const int u0 = c < P.part.N ? P.part.begin(c) : 0, u1 = c < P.part.N ? P.part.begin(c + 1) : 0;
        const int n_chunks = (u1 - u0 + kSChunk - 1) / kSChunk;
        const int wch = max(1, ((kSRLoc - 2) * G + 1) / kSChunk);
        int win_first = 0, win_idx = 0, win_rt0 = u0 / G, cur_rt = -1;
        int k_rt = (u0 + warp) / G, k_g = (u0 + warp) - k_rt * G;
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
        const int pos = *sp.pos;
        if (pos < 0 || pos >= sp.cap) {
          if (tid == 0 && c == 0) atomicOr(sp.status, ST_CTX_FULL);
        } else {
          const int P_eff = attn_splits(pos + 1, sp.P);
          AttnParams a{};
          a.q_dim = sp.q_dim;
          a.kv_dim = sp.kv_dim;
          a.Hkv = sp.Hkv;
          a.P = sp.P;
          a.rope = sp.rope;
          a.rope_neox = sp.rope_neox;
          a.q_norm = P.q_norm;
          a.k_norm = P.k_norm;
          a.eps = sp.eps;
          a.kc = sp.k_base + (size_t)P.layer * sp.layer_stride;
          a.vc = sp.v_base + (size_t)P.layer * sp.layer_stride;
          a.cap = sp.cap;
          a.part = sp.attn_part;
          a.counter = sp.attn_cnt;
          a.out = sp.obuf;
          a.status = sp.status;
          const float* qp = P.qkv_part;
          const int qS = P.qkv_S;
          for (int item = c; item < sp.Hkv * P_eff; item += N)
            attention_item<GQ, HD, kSWarps, ConsumerSync>(a, item / P_eff, item % P_eff, P_eff, pos, sm.u.a,
                                                         [&](int row) {
                                                           const float* src = qp + ((size_t)(row >> 5) * qS) * 32 + (row & 31);
                                                           float x = __ldcg(src);
                                                           for (int j = 1; j < qS; ++j) x += __ldcg(src + j * 32);
                                                           return x;
                                                         });
        }
      } else {
        // ---------------- logits = sum of LM-head partials; greedy choice
        const int V = P.vocab;
        const int r0 = (int)((int64_t)V * c / N), r1 = (int)((int64_t)V * (c + 1) / N);
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        bool nan = false;
        for (int r = r0 + tid; r < r1; r += kSWarps * 32) {
          const float* src = P.lm_part + ((size_t)(r >> 5) * P.lm_S) * 32 + (r & 31);
          float y = __ldcg(src);
          for (int j = 1; j < P.lm_S; ++j) y += __ldcg(src + j * 32);
          sp.logits[r] = y;
          if (y != y) nan = true;
          else if (better(y, r, bv, bi)) { bv = y; bi = r; }
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
          for (int k = tid; k < N; k += kSWarps * 32) {
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
