// Batched decode step (one token for each of M <= 32 sequences) for sm_103a.
//
// The 4-bit matvec of the batch-1 step becomes a skinny GEMM Y[M][rows] =
// X[M][K] W^T. bgemv_kernel: a CTA owns RT_B row tiles (32 rows each) and a
// contiguous range of K units; chunk by chunk it stages the weight units with
// 1-D bulk copies and the normalised input tile, transposed to [k][token], in
// shared memory. Each lane owns a 4-row x 8-token register tile, so every
// weight is dequantised once and used for 8 tokens, every input value for 4
// rows. Arithmetic stays fp32 (exact dequantisation, fp32 accumulation, as in
// the batch-1 path). When K is split over several CTAs the last CTA of a row
// block to arrive adds the partials in CTA order and runs the epilogue
// (store, residual, SwiGLU, or logits with the per-sequence greedy choice).
#pragma once
#include "kernels.cuh"

namespace llmq {

constexpr int kBWarps = 8;
constexpr int kBThreads = kBWarps * 32;
constexpr int kBM = 32;  // tokens per step (sequences), padded to 32

struct BGemvParams {
  const uint8_t* units;    // [n_rt][G] units
  int n_rt, G, K, rows, bf16, unit_bytes, epu;
  int M;                   // live tokens (<= 32)
  int rtb, kc;             // row tiles per CTA, units per chunk (per row tile)
  int ks;                  // K splits (CTAs per row block)
  // input: X [M][K] fp32 (+ optional RMSNorm per token)
  const float* x;
  const float* norm_w;
  float eps;
  // output
  int epi;                 // EPI_STORE / EPI_RESID / EPI_SWIGLU / EPI_LOGITS
  float* out;              // [M][out_cols]
  int out_cols;
  const float* resid;      // [M][rows] (EPI_RESID)
  float* part;             // [ks][M][rows] partials
  int* counters;           // [n_rt / rtb] arrival counters (zero between launches)
  // EPI_LOGITS: per-token best over the row blocks, then the greedy choice
  float* cand_v;           // [M][n_blocks]
  int* cand_i;
  int* gcounter;           // zero between launches
  int* tok_io;             // [M] next-token input of each sequence
  int* argmax_out;         // [M]
  int* pos;                // [M] positions, advanced by one
  int* status;
};

// Dynamic shared memory of one CTA: per stage RT_B*kc units + [kc*epu][32] inputs.
__host__ __device__ inline size_t bgemv_stage_bytes(int rtb, int kc, int unit_bytes, int epu) {
  return (size_t)rtb * kc * unit_bytes + (size_t)kc * epu * kBM * 4;
}

template <bool BF16>
__global__ void __launch_bounds__(kBThreads) bgemv_kernel(const BGemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float s_inv[kBM];
  __shared__ uint64_t s_bar;
  __shared__ int s_last;
  __shared__ float s_bv[kBWarps][kBM];
  __shared__ int s_bi[kBWarps][kBM];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_blocks = p.n_rt / p.rtb;
  const int blk = blockIdx.x / p.ks, ksi = blockIdx.x % p.ks;
  const int g0 = (int)((int64_t)p.G * ksi / p.ks), g1 = (int)((int64_t)p.G * (ksi + 1) / p.ks);
  const int rt0 = blk * p.rtb;
  uint8_t* wbuf = smem;
  float* xbuf = reinterpret_cast<float*>(smem + (size_t)p.rtb * p.kc * p.unit_bytes);  // [kc*epu][32]
  float* red = xbuf;  // reused after the last chunk: [kBWarps][32 lanes][32]

  if (tid == 0) {
    mbar_init(&s_bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();

  // ---- RMSNorm factor per token (the whole row of X), 8 threads per token
  if (p.norm_w) {
    const int m = tid >> 3, sub = tid & 7;
    float ss = 0.f;
    if (m < p.M) {
      const float4* xr = reinterpret_cast<const float4*>(p.x + (size_t)m * p.K);
      for (int i = sub; i < p.K / 4; i += 8) {
        const float4 v = __ldcg(xr + i);
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
      }
    }
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (sub == 0) s_inv[m] = 1.0f / sqrtf(ss / (float)p.K + p.eps);
  }
  __syncthreads();

  // lane tile: rows 4*rg .. 4*rg+3 of the warp's row tile, tokens 8*tg .. 8*tg+7
  const int rg = lane >> 2, tg = lane & 3;
  const int rt_loc = warp % p.rtb, wsub = warp / p.rtb, wstride = kBWarps / p.rtb;
  float acc[4][8];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  uint32_t phase = 0;
  bool ok = true;
  for (int ga = g0; ga < g1 && ok; ga += p.kc) {
    const int nk = min(p.kc, g1 - ga);
    // stage the weight units of every row tile of the block (one bulk copy per row tile)
    if (tid == 0) {
      mbar_expect_tx(&s_bar, p.rtb * nk * p.unit_bytes);
      for (int r = 0; r < p.rtb; ++r)
        bulk_g2s(wbuf + (size_t)r * p.kc * p.unit_bytes, p.units + ((size_t)(rt0 + r) * p.G + ga) * p.unit_bytes,
                 nk * p.unit_bytes, &s_bar, policy_evict_first());
    }
    // stage the (normalised) inputs transposed: xbuf[k][token]
    const int kw = nk * p.epu, kbase = ga * p.epu;
    for (int i = tid; i < kBM * (kw / 4); i += kBThreads) {
      const int m = i % kBM, k4 = i / kBM;  // token fastest: conflict-free transposed stores
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (m < p.M) {
        v = __ldcg(reinterpret_cast<const float4*>(p.x + (size_t)m * p.K + kbase) + k4);
        if (p.norm_w) {
          const float4 w = __ldg(reinterpret_cast<const float4*>(p.norm_w + kbase) + k4);
          const float inv = s_inv[m];
          v = make_float4(v.x * inv * w.x, v.y * inv * w.y, v.z * inv * w.z, v.w * inv * w.w);
        }
      }
      xbuf[(4 * k4 + 0) * kBM + m] = v.x;
      xbuf[(4 * k4 + 1) * kBM + m] = v.y;
      xbuf[(4 * k4 + 2) * kBM + m] = v.z;
      xbuf[(4 * k4 + 3) * kBM + m] = v.w;
    }
    __syncthreads();
    ok = __syncthreads_and(mbar_wait(&s_bar, phase, p.status));  // uniform across the CTA
    phase ^= 1;
    // ---- units of this warp: row tile rt_loc, units wsub, wsub + wstride, ...
    if (ok) {
      for (int u = wsub; u < nk; u += wstride) {
        const uint8_t* ub = wbuf + ((size_t)rt_loc * p.kc + u) * p.unit_bytes;
        const float* xu = xbuf + (size_t)u * p.epu * kBM + tg * 8;
        if (!BF16) {
          float s_[4], m_[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 sm2 = __half22float2(*reinterpret_cast<const __half2*>(ub + 1024 + (4 * rg + i) * 4));
            s_[i] = sm2.x;
            m_[i] = sm2.y;
          }
#pragma unroll
          for (int wd = 0; wd < 8; ++wd) {  // word wd: inputs 32h+8k' + {0..3} (lo) and + {4..7} (hi)
            const int h = wd >> 2, kq = wd & 3;
            float wv[4][8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t v = *reinterpret_cast<const uint32_t*>(ub + (h * 32 + 4 * rg + i) * 16 + 4 * kq);
#pragma unroll
              for (int b = 0; b < 4; ++b) {
                const uint32_t a = __byte_perm(v, 0x4B000000u, 0x7650 + b);
                const float A = __uint_as_float(a), B = __uint_as_float(a & 0xFFFFFFF0u);
                wv[i][b] = fmaf(s_[i], A - B, m_[i]);                               // low nibble
                wv[i][4 + b] = fmaf(s_[i], (B - 8388608.0f) * 0.0625f, m_[i]);     // high nibble
              }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float* xk = xu + (h * 32 + kq * 8 + e) * kBM;
              const float4 xa = *reinterpret_cast<const float4*>(xk);
              const float4 xb = *reinterpret_cast<const float4*>(xk + 4);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                fma2(acc[i][0], acc[i][1], wv[i][e], wv[i][e], xa.x, xa.y);
                fma2(acc[i][2], acc[i][3], wv[i][e], wv[i][e], xa.z, xa.w);
                fma2(acc[i][4], acc[i][5], wv[i][e], wv[i][e], xb.x, xb.y);
                fma2(acc[i][6], acc[i][7], wv[i][e], wv[i][e], xb.z, xb.w);
              }
            }
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < 2; ++kk) {  // inputs 8kk .. 8kk+7
            float wv[4][8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint4 c = *reinterpret_cast<const uint4*>(ub + (kk * 32 + 4 * rg + i) * 16);
              const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
              for (int b = 0; b < 4; ++b) {
                wv[i][2 * b] = __uint_as_float(cw[b] << 16);
                wv[i][2 * b + 1] = __uint_as_float(cw[b] & 0xFFFF0000u);
              }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float* xk = xu + (kk * 8 + e) * kBM;
              const float4 xa = *reinterpret_cast<const float4*>(xk);
              const float4 xb = *reinterpret_cast<const float4*>(xk + 4);
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                fma2(acc[i][0], acc[i][1], wv[i][e], wv[i][e], xa.x, xa.y);
                fma2(acc[i][2], acc[i][3], wv[i][e], wv[i][e], xa.z, xa.w);
                fma2(acc[i][4], acc[i][5], wv[i][e], wv[i][e], xb.x, xb.y);
                fma2(acc[i][6], acc[i][7], wv[i][e], wv[i][e], xb.z, xb.w);
              }
            }
          }
        }
      }
    }
    __syncthreads();  // the buffers are restaged by the next chunk
  }
  if (!ok) return;  // every wait is bounded; the status word carries the timeout

  // ---- each warp's tile -> shared memory (the input staging is no longer needed)
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) red[(warp * 32 + lane) * 32 + i * 8 + j] = acc[i][j];
  __syncthreads();

  // element (r, m) of the block (r < rtb*32 rows, m < 32 tokens) sits in lane
  // (r%32)/4*4 + m/8, slot (r%4)*8 + m%8 of every warp w with w % rtb == r/32
  auto cta_sum = [&](int r, int m) {
    const int rl = r >> 5, rr = r & 31;
    const int ln = (rr >> 2) * 4 + (m >> 3), slot = (rr & 3) * 8 + (m & 7);
    float s = 0.f;
    for (int w = rl; w < kBWarps; w += p.rtb) s += red[(w * 32 + ln) * 32 + slot];
    return s;
  };
  const int rows_blk = p.rtb * 32, row0 = rt0 * 32, rows_pad = p.n_rt * 32;
  const int m = tid & 31, rstep = kBThreads / 32;  // thread: token m, rows tid/32, +8, ...
  bool last = true;
  if (p.ks > 1) {
    for (int r = tid >> 5; r < rows_blk; r += rstep)
      p.part[((size_t)ksi * kBM + m) * rows_pad + row0 + r] = cta_sum(r, m);
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(&p.counters[blk], 1) == p.ks - 1;
    __syncthreads();
    last = s_last;
    if (!last) return;
    __threadfence();
  }
  // final value of (r, m): this CTA's sum, or the K-split partials in CTA order
  auto value = [&](int r, int mm) {
    if (p.ks == 1) return cta_sum(r, mm);
    float s = 0.f;
    for (int j = 0; j < p.ks; ++j) s += __ldcg(p.part + ((size_t)j * kBM + mm) * rows_pad + row0 + r);
    return s;
  };
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  bool nan = false;
  if (m < p.M) {
    for (int r = tid >> 5; r < rows_blk; r += rstep) {
      const int row = row0 + r;
      if (p.epi == EPI_SWIGLU) {  // row tile t: 16 gate rows, then their 16 up rows
        if ((r & 31) < 16) {
          const float g = value(r, m), u = value(r + 16, m);
          p.out[(size_t)m * p.out_cols + (row >> 5) * 16 + (row & 15)] = silu(g) * u;
        }
        continue;
      }
      if (row >= p.rows) continue;
      const float y = value(r, m);
      if (p.epi == EPI_RESID) {
        p.out[(size_t)m * p.out_cols + row] = __ldcg(p.resid + (size_t)m * p.out_cols + row) + y;
      } else {
        p.out[(size_t)m * p.out_cols + row] = y;
        if (p.epi == EPI_LOGITS) {
          if (y != y) nan = true;
          else if (better(y, row, bv, bi)) { bv = y; bi = row; }
        }
      }
    }
  }
  if (p.ks > 1 && tid == 0) p.counters[blk] = 0;
  if (p.epi != EPI_LOGITS) return;
  // ---- greedy choice per sequence: best of this block, then over all blocks
  if (nan) atomicOr(p.status, ST_NAN);
  s_bv[warp][m] = bv;
  s_bi[warp][m] = bi;
  __syncthreads();
  if (tid < kBM) {
    float b2 = s_bv[0][tid];
    int i2 = s_bi[0][tid];
    for (int w = 1; w < kBWarps; ++w)
      if (better(s_bv[w][tid], s_bi[w][tid], b2, i2)) { b2 = s_bv[w][tid]; i2 = s_bi[w][tid]; }
    p.cand_v[(size_t)tid * n_blocks + blk] = b2;
    p.cand_i[(size_t)tid * n_blocks + blk] = i2;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(p.gcounter, 1) == n_blocks - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // warp w handles sequences w, w+8, ...; lanes stride over the blocks
  for (int q = warp; q < p.M; q += kBWarps) {
    float b2 = -INFINITY;
    int i2 = 0x7fffffff;
    for (int k = lane; k < n_blocks; k += 32) {
      const float v = __ldcg(p.cand_v + (size_t)q * n_blocks + k);
      const int ix = __ldcg(p.cand_i + (size_t)q * n_blocks + k);
      if (better(v, ix, b2, i2)) { b2 = v; i2 = ix; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, b2, o);
      const int oi = __shfl_xor_sync(0xffffffffu, i2, o);
      if (better(ov, oi, b2, i2)) { b2 = ov; i2 = oi; }
    }
    if (lane == 0) {
      if (i2 < 0 || i2 >= p.rows) i2 = 0;  // every logit NaN (status already says so)
      p.argmax_out[q] = i2;
      p.tok_io[q] = i2;
      p.pos[q] = p.pos[q] + 1;
    }
  }
  if (tid == 0) *p.gcounter = 0;
}

// x[m][:] = embedding row of token[m] (fp32 or bf16 table)
struct BEmbedParams {
  const void* embed;
  int bf16, dim, vocab, M;
  const int* tok;
  float* x;
  int* status;
};

__global__ void __launch_bounds__(256) bembed_kernel(const BEmbedParams p) {
  pdl_trigger();
  pdl_wait();
  const int m = blockIdx.x;
  int t = p.tok[m];
  if (t < 0 || t >= p.vocab) {
    if (threadIdx.x == 0) atomicOr(p.status, ST_BAD_TOKEN);
    t = 0;
  }
  for (int i = threadIdx.x; i < p.dim; i += 256)
    p.x[(size_t)m * p.dim + i] = p.bf16 ? bf16_bits_to_f32(static_cast<const uint16_t*>(p.embed)[(size_t)t * p.dim + i])
                                        : static_cast<const float*>(p.embed)[(size_t)t * p.dim + i];
}

// Flash-decoding attention of every sequence of the batch: grid (split, kv head, sequence).
struct BAttnParams {
  AttnParams a;           // per-sequence fields are offset below
  const float* qkv;       // [M][q_dim + 2 kv_dim]
  int qkv_cols, o_cols;
  const int* pos;         // [M]
  size_t seq_kv_stride;   // cache elements per sequence
  size_t part_stride;     // attention partial floats per sequence
};

template <int GQ, int HD>
__global__ void __launch_bounds__(kAttnThreads) battention_kernel(const BAttnParams bp) {
  constexpr int NW = kAttnThreads / 32;
  __shared__ __align__(16) AttnSmem<GQ, HD, NW> sm;
  pdl_trigger();
  pdl_wait();
  const int g = blockIdx.y, split = blockIdx.x, b = blockIdx.z;
  AttnParams p = bp.a;
  const int pos = bp.pos[b];
  if (pos < 0 || pos >= p.cap) {
    if (threadIdx.x == 0 && split == 0 && g == 0) atomicOr(p.status, ST_CTX_FULL);
    return;
  }
  const int P_eff = attn_splits(pos + 1, p.P);
  if (split >= P_eff) return;
  p.kc += (size_t)b * bp.seq_kv_stride;
  p.vc += (size_t)b * bp.seq_kv_stride;
  p.part += (size_t)b * bp.part_stride;
  p.counter += (size_t)b * p.Hkv;
  p.out += (size_t)b * bp.o_cols;
  const float* q = bp.qkv + (size_t)b * bp.qkv_cols;
  attention_item<GQ, HD, NW, CtaSync>(p, g, split, P_eff, pos, sm, [&](int row) { return __ldcg(q + row); });
}

}  // namespace llmq
