// Batched decode step (one token for each of M <= 32 sequences) for sm_103a.
//
// The 4-bit matvec of the batch-1 step becomes a skinny GEMM Y[M][rows] =
// X[M][K] W^T. bgemv_kernel: a CTA owns RT_B row tiles (32 rows each) and a
// contiguous range of K units; chunk by chunk it stages the weight units with
// 1-D bulk copies and the normalised inputs in shared memory.
//   * 4-bit units run on the tensor cores (mma.sync m16n8k16, fp16, fp32
//     accumulation): the 4-bit codes become exact fp16 integers, the inputs
//     are bf16 high parts and remainders (64 columns: 32 tokens x 2, a
//     16-bit-mantissa input), and each group's fp16 scale and min are
//     applied to the fp32 MMA result: y = s * sum_k q_k x_k + m * sum_k x_k
//     (the group sums of x by one more MMA against a block of ones).
//     Warp w owns 16 rows of one row tile (with several warps per 16 rows
//     when the block has fewer row tiles, each taking every wp-th unit).
//   * bf16 units (the tied LM head): the same with bf16 operands; the weight
//     fragments are single ldmatrix loads and the inputs are split into bf16
//     high parts and remainders (16-bit mantissa).
// Inputs arrive staged: the producer of a GEMV's input (the embedding, an
// epilogue below, the attention merge) writes it once as XL[64][K], bf16
// high parts of the 32 tokens then their remainders, of x' = x * w with the
// RMSNorm weights w already applied; the consumer copies its rows as they
// are and multiplies each token's result by 1/rms(x) in its epilogue.
// When K is split over several CTAs the last CTA of a row block to arrive
// adds the partials in CTA order and runs the epilogue (store, residual,
// SwiGLU, or logits with the per-sequence greedy choice).
#pragma once
#include <type_traits>

#include "kernels.cuh"
#include "attn_mma.cuh"

namespace llmq {

constexpr int kBWarps = 8;
constexpr int kBThreads = kBWarps * 32;
constexpr int kBM = 32;  // tokens per step (sequences), padded to 32
constexpr int kQKC = 4;  // 4-bit units per chunk (256 inputs) of the tensor-core path
constexpr int kBKsMax = 6;  // K splits (CTAs per row block) at most

struct BGemvParams {
  const uint8_t* units;    // [n_rt][G] units
  int n_rt, G, K, rows, bf16, unit_bytes, epu;
  int M;                   // live tokens (<= 32)
  int rtb, kc;             // row tiles per CTA, units per chunk (per row tile)
  int ks;                  // K splits (CTAs per row block)
  // input: XL [64][K] (see above); with ss_in, RMSNorm: each token's result
  // is scaled by 1/rms(x), from ss_n partial sums of squares ss_in[b * 32 + m]
  const uint16_t* xl;
  const float* ss_in;
  int ss_n;
  float eps;
  // output
  int epi;                 // EPI_STORE / EPI_RESID / EPI_SWIGLU / EPI_LOGITS
  float* out;              // [M][out_cols]
  int out_cols;
  const float* resid;      // [M][rows] (EPI_RESID)
  float* ss_out;           // EPI_RESID: [n_blocks][32] sums of squares of the written rows
  uint16_t* out_hl;        // EPI_RESID / EPI_SWIGLU: the output staged for the next GEMV, XL [64][out_cols]
  const float* out_norm;   // RMSNorm weights that the next GEMV applies to it (null: none)
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

// Dynamic shared memory of one CTA: two buffers of RT_B*kc units (256 inputs
// per row tile) and two of the chunk's staged inputs [64][256+8] halves; after
// the last chunk the per-warp results [8][32][20] fp32.
__host__ __device__ inline size_t bgemv_stage_bytes(int rtb, int kc, int unit_bytes, int epu) {
  const size_t w = (size_t)2 * rtb * kc * unit_bytes;  // two alternating weight buffers
  const size_t x = (size_t)2 * 2 * kBM * (256 + 8) * 2;  // two alternating input buffers
  const size_t red = (size_t)kBWarps * kBM * 20 * 4;
  return (w + x) > red ? (w + x) : red;
}

// Two 4-bit codes of a unit word -> fp16 pair (exact integers 0..15): the
// nibbles sit at bit `sh` and `sh + 8` of w; placed under the exponent of
// 1024 (0x6400) they read 1024 + q, and subtracting 1024 is exact.
__device__ __forceinline__ uint32_t q4_pair_f16(uint32_t w, int sh) {
  uint32_t v = __byte_perm(w >> sh, 0u, 0x4140u);  // [byte0, 0, byte1, 0]
  v = (v & 0x000F000Fu) | 0x64006400u;
  __half2 h = *reinterpret_cast<const __half2*>(&v);
  h = __hsub2(h, __float2half2_rn(1024.f));
  return *reinterpret_cast<const uint32_t*>(&h);
}
// The same as a bf16 pair: under the exponent of 128 (0x4300) the nibble q
// reads 128 + q (7 mantissa bits: exact), and subtracting 128 is exact.
__device__ __forceinline__ uint32_t q4_pair_bf16(uint32_t w, int sh) {
  uint32_t v = __byte_perm(w >> sh, 0u, 0x4140u);
  v = (v & 0x000F000Fu) | 0x43004300u;
  __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&v);
  h = __hsub2(h, __float2bfloat162_rn(128.f));
  return *reinterpret_cast<const uint32_t*>(&h);
}
// Token m's value v at column col of a staged input XL [64][K]: the bf16 high
// part in row m, the bf16 remainder (v - high, rounded) in row 32 + m.
__device__ __forceinline__ void store_hl(uint16_t* xl, int K, int m, int col, float v) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  xl[(size_t)m * K + col] = __bfloat16_as_ushort(h);
  xl[(size_t)(kBM + m) * K + col] = __bfloat16_as_ushort(__float2bfloat16_rn(v - __bfloat162float(h)));
}

template <bool BF16>
__global__ void __launch_bounds__(kBThreads, 2) bgemv_kernel(const BGemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float s_inv[kBM];
  __shared__ uint64_t s_bar[2];
  __shared__ int s_last;
  __shared__ float s_bv[kBWarps][kBM];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_blocks = p.n_rt / p.rtb;
  const int blk = blockIdx.x / p.ks, ksi = blockIdx.x % p.ks;
  const int g0 = (int)((int64_t)p.G * ksi / p.ks), g1 = (int)((int64_t)p.G * (ksi + 1) / p.ks);
  const int rt0 = blk * p.rtb;
  constexpr int KW = 256;          // inputs per chunk
  constexpr int XS = KW + 8;       // staged input row (halves): conflict-free ldmatrix rows
  constexpr int EPU = BF16 ? kBF16UnitCols : 64;
  uint8_t* wbuf = smem;
  // inputs of a chunk: xh[token][k] bf16 high parts, xh[32 + token][k] the remainders (two buffers)
  uint16_t* xh = reinterpret_cast<uint16_t*>(smem + (size_t)2 * p.rtb * p.kc * p.unit_bytes);
  constexpr size_t XB = (size_t)2 * kBM * (KW + 8);  // halves per input buffer

  // the weight units of every row tile of the block (one bulk copy per row
  // tile); weights do not depend on the previous kernel: the first chunk is
  // requested before waiting on it
  const size_t wchunk = (size_t)p.rtb * p.kc * p.unit_bytes;  // one weight buffer (two, alternating)
  auto stage_weights = [&](int ga) {
    const int nk = min(p.kc, g1 - ga), b = ((ga - g0) / p.kc) & 1;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // earlier reads of this buffer
    mbar_expect_tx(&s_bar[b], p.rtb * nk * p.unit_bytes);
    for (int r = 0; r < p.rtb; ++r) {
      // (checked build: an index outside the stream copies its first units instead)
      const bool okc = in_bounds(p.status, rt0 + r < p.n_rt && ga + nk <= p.G);
      bulk_g2s(wbuf + b * wchunk + (size_t)r * p.kc * p.unit_bytes,
               p.units + (okc ? ((size_t)(rt0 + r) * p.G + ga) * p.unit_bytes : 0), nk * p.unit_bytes, &s_bar[b],
               policy_evict_first());
    }
  };
  if (tid == 0) {
    mbar_init(&s_bar[0], 1);
    mbar_init(&s_bar[1], 1);
    mbar_fence_init();
    stage_weights(g0);
    if (g0 + p.kc < g1) stage_weights(g0 + p.kc);
  }
  __syncthreads();
  pdl_trigger();
  pdl_wait();

  // a chunk's inputs, copied as they are (cp.async, 16 B = 8 inputs of a
  // token's high parts or remainders) into input buffer bi; absent tokens
  // and columns past the chunk read zero. The first chunk's copies go out in
  // the same round trip as the RMSNorm statistics.
  constexpr int NL = kBM * (KW / 8) / kBThreads;  // copies per thread and half (k fastest: coalesced)
  static_assert(kBThreads % (KW / 8) == 0, "a thread stages one input column (k8) for NL tokens");
  const int k8 = tid % (KW / 8);
  auto load_inputs = [&](int ga, int bi) {
    const int kw = min(p.kc, g1 - ga) * EPU, kbase = ga * EPU;
#pragma unroll
    for (int it = 0; it < NL; ++it) {
      const int m = (tid + it * kBThreads) / (KW / 8);
#pragma unroll
      for (int hl = 0; hl < 2; ++hl) {
        uint16_t* dst = xh + bi * XB + (size_t)(hl * kBM + m) * XS + 8 * k8;
        if (m < p.M && k8 < kw / 8) cp_async16(dst, p.xl + (size_t)(hl * kBM + m) * p.K + kbase + 8 * k8);
        else *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  };
  load_inputs(g0, 0);
  cp_async_commit();

  // ---- RMSNorm factor per token from the producer's partial sums of squares
  // (thread: token tid % 32, partials tid/32, +8, ...; added in a fixed order)
  if (p.ss_in) {
    const int m = tid & 31, sub = tid >> 5;
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = ldcg1_if(p.ss_in + (size_t)(sub + 8 * j) * kBM + m, sub + 8 * j < p.ss_n);
    float ss = ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
    for (int b = sub + 64; b < p.ss_n; b += 8) ss += __ldcg(p.ss_in + (size_t)b * kBM + m);  // > 64 partials
    s_bv[sub][m] = ss;
    __syncthreads();
    if (tid < kBM) {
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < kBWarps; ++w) t += s_bv[w][tid];
      s_inv[tid] = 1.0f / sqrtf(t / (float)p.K + p.eps);
    }
  }
  __syncthreads();

  // warp -> 16 rows (row tile rt_q, half 16*(pair&1)) x every wp-th unit of the chunk;
  // lane (g, t) holds rows R0 = 16*(pair&1) + g, R0 + 8 and tokens 8nt + 2t + e
  const int wp = kBWarps / (2 * p.rtb), pair = warp / wp, usub = warp % wp;
  const int rt_q = pair >> 1, mt = pair & 1, R0 = 16 * mt + (lane >> 2), t = lane & 3;
  const int r8 = lane & 7, mi = lane >> 3;
  const int sh = 16 * (t & 1) + 4 * (t >> 1);  // 4-bit: bit of input 2t within its code word
  float qacc[4][2][2];
#pragma unroll
  for (int i = 0; i < 4; ++i) qacc[i][0][0] = qacc[i][0][1] = qacc[i][1][0] = qacc[i][1][1] = 0.f;

  bool ok = true;
  int n_issued = min(2, (g1 - g0 + p.kc - 1) / p.kc), ci_fail = 0;  // weight chunks requested (thread 0)
  for (int ga = g0, ci = 0; ga < g1 && ok; ga += p.kc, ++ci) {
    const int nk = min(p.kc, g1 - ga);
    const uint8_t* wb = wbuf + (ci & 1) * wchunk;
    const uint16_t* xb = xh + (ci & 1) * XB;
    if (ga + p.kc < g1) load_inputs(ga + p.kc, (ci + 1) & 1);  // in flight while this chunk computes
    cp_async_commit();
    cp_async_wait_group<1>();  // this chunk's inputs
    ok = __syncthreads_and(mbar_wait(&s_bar[ci & 1], (ci >> 1) & 1, p.status));  // uniform across the CTA
    ci_fail = ci;
    if (ok) {
      for (int u = usub; u < nk; u += wp) {
        float d[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) d[nt][0] = d[nt][1] = d[nt][2] = d[nt][3] = 0.f;
        if constexpr (!BF16) {
          // ds[j]: the group's input sums (high parts + remainders) of tokens 8j .. 8j+7, by MMAs
          // against a block of ones (every row of the result holds them)
          float ds[4][4];
#pragma unroll
          for (int j = 0; j < 4; ++j) ds[j][0] = ds[j][1] = ds[j][2] = ds[j][3] = 0.f;
          const uint8_t* ub = wb + ((size_t)rt_q * p.kc + u) * p.unit_bytes;
          // rows R0 and R0 + 8: 16 B of codes per input half (inputs 0-31, 32-63)
          const uint4 c00 = *reinterpret_cast<const uint4*>(ub + R0 * 16);
          const uint4 c01 = *reinterpret_cast<const uint4*>(ub + (32 + R0) * 16);
          const uint4 c10 = *reinterpret_cast<const uint4*>(ub + (R0 + 8) * 16);
          const uint4 c11 = *reinterpret_cast<const uint4*>(ub + (32 + R0 + 8) * 16);
          const float2 sm0 = __half22float2(*reinterpret_cast<const __half2*>(ub + 1024 + 4 * R0));
          const float2 sm1 = __half22float2(*reinterpret_cast<const __half2*>(ub + 1024 + 4 * (R0 + 8)));
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            // inputs 16ks + 2t(+1) and +8 sit in words 2(ks%2) and 2(ks%2)+1 of input half ks/2
            const uint4 w0 = ks < 2 ? c00 : c01, w1 = ks < 2 ? c10 : c11;
            const uint32_t w0a = (ks & 1) ? w0.z : w0.x, w0b = (ks & 1) ? w0.w : w0.y;
            const uint32_t w1a = (ks & 1) ? w1.z : w1.x, w1b = (ks & 1) ? w1.w : w1.y;
            const uint32_t a[4] = {q4_pair_bf16(w0a, sh), q4_pair_bf16(w1a, sh), q4_pair_bf16(w0b, sh),
                                   q4_pair_bf16(w1b, sh)};
            constexpr uint32_t kOne2 = 0x3F803F80u;  // bf16 (1, 1)
            const uint32_t ones[4] = {kOne2, kOne2, kOne2, kOne2};
#pragma unroll
            for (int nt = 0; nt < 8; nt += 2) {
              uint32_t b[4];
              ldsm_x4(b, xb + (size_t)(8 * (nt + (mi >> 1)) + r8) * XS + u * 64 + 16 * ks + 8 * (mi & 1));
              mma_bf16_16816(d[nt], a, b[0], b[1]);
              mma_bf16_16816(d[nt + 1], a, b[2], b[3]);
              mma_bf16_16816(ds[nt & 3], ones, b[0], b[1]);
              mma_bf16_16816(ds[(nt + 1) & 3], ones, b[2], b[3]);
            }
          }
          // y += s * (high + remainder columns) + m * sum(x)
#pragma unroll
          for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float X = ds[nt][e];
              qacc[nt][e][0] = fmaf(sm0.x, d[nt][e] + d[nt + 4][e], fmaf(sm0.y, X, qacc[nt][e][0]));
              qacc[nt][e][1] = fmaf(sm1.x, d[nt][2 + e] + d[nt + 4][2 + e], fmaf(sm1.y, X, qacc[nt][e][1]));
            }
        } else {
          // bf16 unit [k half][row][8 k]: the A fragment of rows 16mt.. is one ldmatrix
          const uint8_t* ub = wb + ((size_t)rt_q * p.kc + u) * p.unit_bytes;
          uint32_t a[4];
          ldsm_x4(a, ub + ((mi >> 1) * 32 + 16 * mt + 8 * (mi & 1) + r8) * 16);
#pragma unroll
          for (int nt = 0; nt < 8; nt += 2) {
            uint32_t b[4];
            ldsm_x4(b, xb + (size_t)(8 * (nt + (mi >> 1)) + r8) * XS + u * 16 + 8 * (mi & 1));
            mma_bf16_16816(d[nt], a, b[0], b[1]);
            mma_bf16_16816(d[nt + 1], a, b[2], b[3]);
          }
#pragma unroll
          for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              qacc[nt][e][0] += d[nt][e] + d[nt + 4][e];
              qacc[nt][e][1] += d[nt][2 + e] + d[nt + 4][2 + e];
            }
        }
      }
    }
    __syncthreads();  // the buffers are restaged by the next chunks
    if (tid == 0 && ok && ga + 2 * p.kc < g1) {
      stage_weights(ga + 2 * p.kc);  // into this chunk's buffer
      ++n_issued;
    }
  }
  if (!ok) {  // every wait is bounded; the status word carries the timeout
    cp_async_wait_all();
    if (tid == 0)  // the weight copies still in flight land (bounded waits) before the CTA leaves
      for (int c = ci_fail; c < n_issued; ++c) mbar_wait(&s_bar[c & 1], (c >> 1) & 1, p.status);
    return;
  }

  // ---- each warp's results -> shared memory [warp][32 tokens][QS] (16 rows,
  // padded: both the fragment stores and the row-contiguous reads below are
  // free of bank conflicts); the staging is no longer needed
  constexpr int QS = 20;
  float* qred = reinterpret_cast<float*>(smem);
  {
    const int rr = lane >> 2;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        qred[(warp * kBM + 8 * nt + 2 * t + e) * QS + rr] = qacc[nt][e][0];
        qred[(warp * kBM + 8 * nt + 2 * t + e) * QS + rr + 8] = qacc[nt][e][1];
      }
  }
  __syncthreads();
  // Sum of this CTA for element (r, m) of the block (r < rtb*32 rows, m < 32
  // tokens): rows 16h .. 16h+15 of row tile rl are the wp warps of pair 2rl + h.
  auto cta_sum = [&](int r, int mm) {
    const int pr = r >> 4, rr = r & 15;
    float v = 0.f;
    for (int w = pr * wp; w < pr * wp + wp; ++w) v += qred[(w * kBM + mm) * QS + rr];
    return v;
  };
  // Epilogue: warp w takes tokens w, w+8, w+16, w+24; lane = row within a row
  // tile, so every global access below is one contiguous 128-B line.
  const int row0 = rt0 * 32, rows_pad = p.n_rt * 32;
  if (p.ks > 1) {
    for (int rl = 0; rl < p.rtb; ++rl)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int mm = warp + 8 * k;
        const float v = cta_sum(rl * 32 + lane, mm);
        if (in_bounds(p.status, ksi < p.ks && row0 + rl * 32 + lane < rows_pad))
          p.part[((size_t)ksi * kBM + mm) * rows_pad + row0 + rl * 32 + lane] = v;
      }
    __syncthreads();
    if (tid == 0) {  // one release for the CTA's partials (ordered after them by the barrier)
      __threadfence();
      s_last = atomicAdd(&p.counters[blk], 1) == p.ks - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
  }
  static_assert(kBKsMax <= 6, "partials of 4 tokens in flight per thread");
  float ssq[4] = {0.f, 0.f, 0.f, 0.f};  // EPI_RESID: sums of squares per token of the warp
  float bv[4];
  int bi[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    bv[k] = -INFINITY;
    bi[k] = 0x7fffffff;
  }
  bool nan = false;
  for (int rl = 0; rl < p.rtb; ++rl) {
    const int r = rl * 32 + lane, row = row0 + r;
    // EPI_RESID: the residual rows, requested with the partials (one round trip)
    float rv[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      rv[k] = ldcg1_if(p.resid + (size_t)(warp + 8 * k) * p.out_cols + row,
                       p.epi == EPI_RESID && warp + 8 * k < p.M && row < p.rows);
    float y[4];
    if (p.ks == 1) {
#pragma unroll
      for (int k = 0; k < 4; ++k) y[k] = cta_sum(r, warp + 8 * k);
    } else {  // the K-split partials of the 4 tokens, all in flight together, added in CTA order
      float pv[4][kBKsMax];
#pragma unroll
      for (int k = 0; k < 4; ++k)
#pragma unroll
        for (int j = 0; j < kBKsMax; ++j)
          pv[k][j] = ldcg1_if(p.part + ((size_t)j * kBM + warp + 8 * k) * rows_pad + row, j < p.ks);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < kBKsMax; ++j) sum += pv[k][j];
        y[k] = sum;
      }
    }
    if (p.ss_in)  // RMSNorm of the input: 1/rms per token on the result
#pragma unroll
      for (int k = 0; k < 4; ++k) y[k] *= s_inv[warp + 8 * k];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int mm = warp + 8 * k;
      if (p.epi == EPI_SWIGLU) {  // lanes 0-15: gate rows; their up rows are lanes 16-31
        const float up = __shfl_down_sync(0xffffffffu, y[k], 16);
        if (mm < p.M && lane < 16) {
          const int col = (row >> 5) * 16 + lane;
          const float av = silu(y[k]) * up;
          if (p.out) p.out[(size_t)mm * p.out_cols + col] = av;
          if (p.out_hl) store_hl(p.out_hl, p.out_cols, mm, col, av);
        }
        continue;
      }
      if (mm >= p.M || row >= p.rows) continue;
      if (p.epi == EPI_RESID) {
        const float xn = rv[k] + y[k];
        p.out[(size_t)mm * p.out_cols + row] = xn;
        if (p.out_hl) store_hl(p.out_hl, p.out_cols, mm, row, p.out_norm ? xn * __ldg(p.out_norm + row) : xn);
        ssq[k] += xn * xn;
      } else {
        p.out[(size_t)mm * p.out_cols + row] = y[k];
        if (p.epi == EPI_LOGITS) {
          if (y[k] != y[k]) nan = true;
          else if (better(y[k], row, bv[k], bi[k])) { bv[k] = y[k]; bi[k] = row; }
        }
      }
    }
  }
  if (p.ks > 1 && tid == 0) p.counters[blk] = 0;
  if (p.epi == EPI_RESID && p.ss_out) {  // per-token partial over this block's rows
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float v = ssq[k];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) p.ss_out[(size_t)blk * kBM + warp + 8 * k] = v;
    }
    return;
  }
  if (p.epi != EPI_LOGITS) return;
  // ---- greedy choice per sequence: best of this block, then over all blocks
  if (nan) atomicOr(p.status, ST_NAN);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv[k], o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi[k], o);
      if (better(ov, oi, bv[k], bi[k])) { bv[k] = ov; bi[k] = oi; }
    }
    if (lane == 0) {
      p.cand_v[(size_t)(warp + 8 * k) * n_blocks + blk] = bv[k];
      p.cand_i[(size_t)(warp + 8 * k) * n_blocks + blk] = bi[k];
    }
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

// ---- the batched LM head over a bf16 table (the tied embedding) ------------
// Persistent: one CTA per SM walks a contiguous range of row tiles with the
// 32-token staged input (XL, above) copied once for the whole launch and
// resident in shared memory; 1/rms scales each logit. Consumer
// warp w owns row tile w of each group of kHWarps and accumulates it over all
// of K (both 16-row halves share the input fragments). A producer warp
// streams the group's units through a ring of kHSlots slots (kHUC units of
// every row tile of the group per slot), running ahead across groups. Each
// warp stores its row tile's logits when it finishes it and keeps the best
// logit of each token; the CTA's best goes to cand_v/cand_i[token][CTA], and
// the last CTA to arrive picks each sequence's greedy choice.
constexpr int kHWarps = 8;                        // consumer warps = row tiles in flight
constexpr int kHThreads = (kHWarps + 1) * 32;     // + the producer warp
constexpr int kHUC = 2;                           // units of each row tile per ring slot
constexpr int kHSlots = 5;
constexpr int kHUnitBytes = 32 * kBF16UnitCols * 2;
constexpr size_t kHSlotBytes = (size_t)kHWarps * kHUC * kHUnitBytes;

// Dynamic shared memory: the ring, then the inputs [64][K+8] halves.
__host__ __device__ inline size_t bhead_smem_bytes(int K) {
  return (size_t)kHSlots * kHSlotBytes + (size_t)2 * kBM * (K + 8) * 2;
}

__device__ __forceinline__ void consumers_sync() {  // the kHWarps consumer warps only
  asm volatile("bar.sync 1, %0;" ::"n"(kHWarps * 32) : "memory");
}

__global__ void __launch_bounds__(kHThreads, 1) bhead_kernel(const BGemvParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t s_full[kHSlots], s_empty[kHSlots];
  __shared__ float s_inv[kBM];
  __shared__ float s_bv[kHWarps][kBM];
  __shared__ int s_bi[kHWarps][kBM];
  __shared__ int s_last, s_fail;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int XS = p.K + 8;  // staged input row (halves): conflict-free ldmatrix rows
  uint8_t* ring = smem;
  uint16_t* xh = reinterpret_cast<uint16_t*>(smem + (size_t)kHSlots * kHSlotBytes);
  const int nc = gridDim.x, c = blockIdx.x;
  const int rt_a = (int)((int64_t)p.n_rt * c / nc), rt_b = (int)((int64_t)p.n_rt * (c + 1) / nc);
  const int n_groups = (rt_b - rt_a + kHWarps - 1) / kHWarps;
  if (tid == 0) {
    for (int i = 0; i < kHSlots; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], kHWarps);
    }
    mbar_fence_init();
    s_fail = 0;
  }
  __syncthreads();

  if (warp == kHWarps) {  // ---- producer: weights only (no wait on the previous kernel)
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      int ci = 0;
      bool live = true;
      for (int gi = 0; gi < n_groups && live; ++gi) {
        const int rt0 = rt_a + gi * kHWarps, nrt = min(kHWarps, rt_b - rt0);
        for (int u0 = 0; u0 < p.G && live; u0 += kHUC, ++ci) {
          const int slot = ci % kHSlots;
          if (ci >= kHSlots) {
            if (!mbar_wait_spin(&s_empty[slot], ((ci / kHSlots) - 1) & 1, p.status)) {
              live = false;
              break;
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the consumers' reads of the slot
          }
          mbar_expect_tx(&s_full[slot], (uint32_t)(nrt * kHUC * kHUnitBytes));
          for (int r = 0; r < nrt; ++r) {
            const bool okc = in_bounds(p.status, rt0 + r < p.n_rt && u0 + kHUC <= p.G);
            bulk_g2s(ring + slot * kHSlotBytes + (size_t)r * kHUC * kHUnitBytes,
                     p.units + (okc ? ((size_t)(rt0 + r) * p.G + u0) * kHUnitBytes : 0), kHUC * kHUnitBytes,
                     &s_full[slot], pol);
          }
        }
      }
      // before leaving, every copy this warp issued has landed (at once on the normal path, where the
      // consumers waited for them; bounded after a timeout): the last chunk of each slot
      for (int c = max(0, ci - kHSlots); c < ci; ++c) mbar_wait(&s_full[c % kHSlots], (c / kHSlots) & 1, p.status);
    }
    return;
  }

  // ---- consumers: RMSNorm factor per token from the producer's partial sums
  // of squares (thread: token tid % 32, partials tid/32, +8, ...; fixed order)
  pdl_trigger();
  pdl_wait();
  if (p.ss_in) {
    const int m = tid & 31, sub = tid >> 5;
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = ldcg1_if(p.ss_in + (size_t)(sub + 8 * j) * kBM + m, sub + 8 * j < p.ss_n);
    float ss = ((v[0] + v[1]) + (v[2] + v[3])) + ((v[4] + v[5]) + (v[6] + v[7]));
    for (int b = sub + 64; b < p.ss_n; b += 8) ss += __ldcg(p.ss_in + (size_t)b * kBM + m);  // > 64 partials
    s_bv[sub][m] = ss;
    consumers_sync();
    if (tid < kBM) {
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < kHWarps; ++w) t += s_bv[w][tid];
      s_inv[tid] = 1.0f / sqrtf(t / (float)p.K + p.eps);
    }
  }
  // the whole staged input, once: 16 B (8 inputs) of a token's high parts or remainders per load
  {
    const int k8n = p.K / 8;
    constexpr int UN = 8;  // loads in flight per thread
    for (int i0 = tid; i0 < 2 * kBM * k8n; i0 += UN * kHWarps * 32) {
      float4 xv[UN];
#pragma unroll
      for (int j = 0; j < UN; ++j) {
        const int i = i0 + j * kHWarps * 32, r = i / k8n, k8 = i - r * k8n;
        xv[j] = ldcg4_if(reinterpret_cast<const float*>(p.xl + (size_t)r * p.K + 8 * k8),
                         i < 2 * kBM * k8n && (r & (kBM - 1)) < p.M);
      }
#pragma unroll
      for (int j = 0; j < UN; ++j) {
        const int i = i0 + j * kHWarps * 32, r = i / k8n, k8 = i - r * k8n;
        if (i < 2 * kBM * k8n) *reinterpret_cast<float4*>(xh + (size_t)r * XS + 8 * k8) = xv[j];
      }
    }
  }
  consumers_sync();

  // lane (g, t): rows 16h + g (+8) of its row tile, tokens 8nt + 2t + e; the
  // accumulators hold the high-part columns (nt < 4) and the remainders (nt >= 4)
  const int g = lane >> 2, t = lane & 3, r8 = lane & 7, mi = lane >> 3;
  float bv[4][2];
  int bi[4][2];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      bv[nt][e] = -INFINITY;
      bi[nt][e] = 0x7fffffff;
    }
  bool ok = true, nan = false;
  int ci = 0;
  for (int gi = 0; gi < n_groups; ++gi) {
    const int rt = rt_a + gi * kHWarps + warp;
    const bool mine = rt < rt_b;
    float d[2][8][4];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) d[h][nt][0] = d[h][nt][1] = d[h][nt][2] = d[h][nt][3] = 0.f;
    for (int u0 = 0; u0 < p.G; u0 += kHUC, ++ci) {
      const int slot = ci % kHSlots;
      if (ok) ok = mbar_wait_spin(&s_full[slot], (ci / kHSlots) & 1, p.status);
      if (ok && mine) {
        const uint8_t* wb = ring + slot * kHSlotBytes + (size_t)warp * kHUC * kHUnitBytes;
#pragma unroll
        for (int uu = 0; uu < kHUC; ++uu) {
          uint32_t bx[4][4];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            ldsm_x4(bx[q], xh + (size_t)(8 * (2 * q + (mi >> 1)) + r8) * XS + (u0 + uu) * kBF16UnitCols + 8 * (mi & 1));
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            // bf16 unit [k half][row][8 k]: the A fragment of rows 16h .. 16h+15 is one ldmatrix
            uint32_t a[4];
            ldsm_x4(a, wb + (size_t)uu * kHUnitBytes + ((mi >> 1) * 32 + 16 * h + 8 * (mi & 1) + r8) * 16);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              mma_bf16_16816(d[h][2 * q], a, bx[q][0], bx[q][1]);
              mma_bf16_16816(d[h][2 * q + 1], a, bx[q][2], bx[q][3]);
            }
          }
        }
      }
      __syncwarp();
      if (ok && lane == 0) mbar_arrive(&s_empty[slot]);
    }
    if (!ok || !mine) continue;
    // this row tile's logits (4 tokens x 8 consecutive rows per store: whole 32-B sectors)
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int row = rt * 32 + 16 * h + 8 * hh + g;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int mm = 8 * nt + 2 * t + e;
            float y = d[h][nt][2 * hh + e] + d[h][nt + 4][2 * hh + e];
            if (mm >= p.M || row >= p.rows) continue;
            if (p.ss_in) y *= s_inv[mm];  // RMSNorm of the input: 1/rms per token
            p.out[(size_t)mm * p.out_cols + row] = y;
            if (y != y) nan = true;
            else if (better(y, row, bv[nt][e], bi[nt][e])) {
              bv[nt][e] = y;
              bi[nt][e] = row;
            }
          }
      }
  }
  // ---- greedy choice: best per token over the lanes of a warp, the warps, then the CTAs
  if (!ok) s_fail = 1;
  if (nan) atomicOr(p.status, ST_NAN);
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {  // lanes of equal t hold the same tokens
        const float ov = __shfl_xor_sync(0xffffffffu, bv[nt][e], o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi[nt][e], o);
        if (better(ov, oi, bv[nt][e], bi[nt][e])) {
          bv[nt][e] = ov;
          bi[nt][e] = oi;
        }
      }
      if (g == 0) {
        s_bv[warp][8 * nt + 2 * t + e] = bv[nt][e];
        s_bi[warp][8 * nt + 2 * t + e] = bi[nt][e];
      }
    }
  consumers_sync();
  if (s_fail) return;  // every consumer warp has passed its last barrier; the status word says why
  const int n_blocks = nc;
  if (warp == 0) {
    float b2 = -INFINITY;
    int i2 = 0x7fffffff;
#pragma unroll
    for (int w = 0; w < kHWarps; ++w)
      if (better(s_bv[w][lane], s_bi[w][lane], b2, i2)) {
        b2 = s_bv[w][lane];
        i2 = s_bi[w][lane];
      }
    p.cand_v[(size_t)lane * n_blocks + c] = b2;
    p.cand_i[(size_t)lane * n_blocks + c] = i2;
  }
  __threadfence();
  consumers_sync();
  if (tid == 0) s_last = atomicAdd(p.gcounter, 1) == n_blocks - 1;
  consumers_sync();
  if (!s_last) return;
  __threadfence();
  // warp w handles sequences w, w+8, ...; lanes stride over the CTAs
  for (int q = warp; q < p.M; q += kHWarps) {
    float b2 = -INFINITY;
    int i2 = 0x7fffffff;
    for (int k = lane; k < n_blocks; k += 32) {
      const float v = __ldcg(p.cand_v + (size_t)q * n_blocks + k);
      const int ix = __ldcg(p.cand_i + (size_t)q * n_blocks + k);
      if (better(v, ix, b2, i2)) {
        b2 = v;
        i2 = ix;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, b2, o);
      const int oi = __shfl_xor_sync(0xffffffffu, i2, o);
      if (better(ov, oi, b2, i2)) {
        b2 = ov;
        i2 = oi;
      }
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
  float* ss_out;         // [32]: sum of squares of each token's row
  uint16_t* x_hl;        // the rows staged for the first GEMV, XL [64][dim], with
  const float* norm_w;   // its RMSNorm weights applied
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
  float ss = 0.f;
  for (int i = threadIdx.x; i < p.dim; i += 256) {
    const float v = p.bf16 ? bf16_bits_to_f32(static_cast<const uint16_t*>(p.embed)[(size_t)t * p.dim + i])
                           : static_cast<const float*>(p.embed)[(size_t)t * p.dim + i];
    p.x[(size_t)m * p.dim + i] = v;
    store_hl(p.x_hl, p.dim, m, i, v * __ldg(p.norm_w + i));
    ss += v * v;
  }
  // sum of squares of the row (the first RMSNorm): warps, then warp sums in order
  __shared__ float s_w[8];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < 8; ++w) t += s_w[w];
    p.ss_out[m] = t;
  }
}

// Flash-decoding attention of every sequence of the batch: grid (split, kv head, sequence).
enum BAttnMode : int { BA_APPEND_ATTEND = 0, BA_APPEND = 1, BA_ATTEND = 2 };

struct BAttnParams {
  AttnParams a;           // per-sequence fields are offset below
  const float* qkv;       // [M][q_dim + 2 kv_dim]
  int qkv_cols, o_cols;
  const int* pos;         // [M] position of each row's token
  const int* seq;         // [M] cache (sequence) of each row, or null: row b uses cache b
  int mode;               // BA_APPEND_ATTEND; or, for several rows of one sequence (a prompt
                          // chunk), BA_APPEND for all rows, then BA_ATTEND over the cache
  size_t seq_kv_stride;   // cache elements per sequence
  size_t part_stride;     // attention partial floats per row
  uint16_t* o_hl;         // the output, staged for the o-projection: XL [64][o_cols]
  int8_t* k8;             // the grouped int8 cache instead of a.kc / a.vc (layer base): codes
  int8_t* v8;
  uint16_t* ks;           // and fp16 scales of each 32 values (layer base; elements / 32)
  uint16_t* vs;
};


#ifndef LLMQ_BATTN_SPLIT_LEN
// Cached positions per split (at most 24 splits per (sequence, kv head)).
// Measured on the 32-sequence workload, bf16 cache: 128 -> 9408, 256 -> 10005,
// 512 -> 10826, 768 -> 10176, 1024 -> 10735 tok/s; again with the bf16 MMAs
// and the one-round-trip GEMV merge, ms per step: 384 -> 2.68, 512 -> 2.56,
// 768 -> 2.76
#define LLMQ_BATTN_SPLIT_LEN 512
#endif
constexpr int kBAttnThreads = 256;

// Shared memory of one batched attention item (sequence, kv head, split) over
// the bf16 cache: each warp streams its own blocks of 16 positions through a
// private stage (bf16 rows as cached, unpadded, chunks permuted by tile_off)
// and keeps its own running softmax state, so no CTA barrier separates two
// blocks (~76 KB for Qwen3's GQ 2, hd 128: 3 CTAs per SM).
template <int GQ, int HD>
struct BAttnWarpSmem {
  static constexpr int NW = kBAttnThreads / 32;
  uint16_t kt[NW][16][HD];
  uint16_t vt[NW][16][HD];
  float cur[GQ + 2][HD];          // q heads (scaled), k, v of this step
  float tres[NW][GQ][HD + 2];     // per warp: the block's o, max, sum; at the end the warp's state
  int is_last;
};
// The same over the grouped int8 cache: a warp's stage holds its block's
// codes widened to fp16 (exact) in the same permuted rows, and their fp16
// group scales (~78 KB for GQ 2, hd 128: 2 CTAs per SM).
template <int GQ, int HD>
struct BAttnWarpSmem8 {
  static constexpr int NW = kBAttnThreads / 32, NG = HD / 32;
  uint16_t kt[NW][16][HD];
  uint16_t vt[NW][16][HD];
  __align__(16) uint16_t ksc[NW][16][NG];
  __align__(16) uint16_t vsc[NW][16][NG];
  float cur[GQ + 2][HD];          // q heads (scaled), k, v of this step (k, v: their codes)
  float cursc[2][NG];             // this step's k, v group scales
  float tres[NW][GQ][HD + 2];
  int is_last;
};
template <int GQ, int HD, bool KV8>
using BAttnSmemT = std::conditional_t<KV8, BAttnWarpSmem8<GQ, HD>, BAttnWarpSmem<GQ, HD>>;

// Flash-decoding attention of every sequence of the batch on the tensor
// cores: grid (split, kv head, sequence), splits of LLMQ_BATTN_SPLIT_LEN
// positions. Warp w takes blocks w, w+8, ... of 16 positions of the split:
// it copies each into its private stage (bf16 rows as cached; int8 codes
// widened to fp16 in the stage), scores all GQ heads on the tensor cores
// (attn_mma.cuh: bf16 operands for the bf16 cache, fp16 for the widened
// codes; the query's fragments packed once per item), folds the block into
// its own running (max, sum, o), and requests its next block as soon as the
// stage has been read. The 8 warp states merge once per
// split, and the last split of a (sequence, kv head) to finish merges the
// splits into the output row.
template <int GQ, int HD, bool KV8>
__global__ void __launch_bounds__(kBAttnThreads) battn_mma_kernel(const BAttnParams bp) {
  using SA = BAttnSmemT<GQ, HD, KV8>;
  constexpr int NT = kBAttnThreads, NW = SA::NW, CH = HD / 8, DPL = HD / 32, NG = HD / 32;
  static_assert(GQ <= 8 && NW == 8, "layout");
  extern __shared__ __align__(16) uint8_t smraw[];
  SA& sa = *reinterpret_cast<SA*>(smraw);
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y, split = blockIdx.x, b = blockIdx.z;
  const AttnParams& a = bp.a;
  const int pos = bp.pos[b];
  if (pos < 0 || pos >= a.cap) {
    if (tid == 0 && split == 0 && g == 0) atomicOr(a.status, ST_CTX_FULL);
    return;
  }
  const int len = pos + 1;
  constexpr int PMAX = 24;  // merge scratch: splits a (sequence, kv head) may have
  const int P_eff = min(min(a.P, PMAX), (len + LLMQ_BATTN_SPLIT_LEN - 1) / LLMQ_BATTN_SPLIT_LEN);
  if (split >= P_eff) return;
  const int t0 = (int)((int64_t)len * split / P_eff), t1 = (int)((int64_t)len * (split + 1) / P_eff);
  const int sb = bp.seq ? bp.seq[b] : b;  // this row's cache
  const size_t cbase = (size_t)sb * bp.seq_kv_stride + (size_t)g * a.cap * HD;
  uint16_t* kc = KV8 ? nullptr : a.kc + cbase;
  uint16_t* vc = KV8 ? nullptr : a.vc + cbase;
  int8_t* kc8 = KV8 ? bp.k8 + cbase : nullptr;  // int8 K/V: codes and group scales
  int8_t* vc8 = KV8 ? bp.v8 + cbase : nullptr;
  uint16_t* ks8 = KV8 ? bp.ks + cbase / 32 : nullptr;
  uint16_t* vs8 = KV8 ? bp.vs + cbase / 32 : nullptr;
  const bool attend = bp.mode != BA_APPEND;
  const bool append = bp.mode == BA_APPEND || (bp.mode == BA_APPEND_ATTEND && split == P_eff - 1);
  const float* qkv = bp.qkv + (size_t)b * bp.qkv_cols;

  // the warp's block: rows tp .. tp+n-1 (n <= 16) of K and V into its stage
  // (async copies). bf16: the rows as cached, rows past n zero. int8: each
  // row's codes into the first HD bytes of its fp16 row, its scales beside;
  // widen() then makes them fp16 in place
  static_assert((CH & (CH - 1)) == 0, "16-B chunks per row: a power of two");
  constexpr int LCH = CH == 8 ? 3 : 4;
  auto stage = [&](int tp) {
    const int n = min(16, t1 - tp);
    if constexpr (KV8) {
      constexpr int C8 = HD / 16, L8 = C8 == 4 ? 2 : 3;
      for (int idx = lane; idx < 2 * 16 * C8; idx += 32) {
        const int kv = idx >= 16 * C8, r = idx - kv * 16 * C8, row = r >> L8, ch = r & (C8 - 1);
        if (row < n && in_bounds(a.status, tp + row < a.cap))
          cp_async16(reinterpret_cast<uint8_t*>(&(kv ? sa.vt : sa.kt)[warp][row][0]) + 16 * ch,
                     (kv ? vc8 : kc8) + (size_t)(tp + row) * HD + 16 * ch);
      }
      const int kv = lane >> 4, row = lane & 15;  // one row's scales per lane
      if (row < n && in_bounds(a.status, tp + row < a.cap))
        cp_async_small<2 * NG>(&(kv ? sa.vsc : sa.ksc)[warp][row][0], (kv ? vs8 : ks8) + (size_t)(tp + row) * NG);
    } else {
      for (int idx = lane; idx < 2 * 16 * CH; idx += 32) {
        const int kv = idx >= 16 * CH, r = idx - kv * 16 * CH, row = r >> LCH, ch = r & (CH - 1);
        uint16_t* dst = &(kv ? sa.vt : sa.kt)[warp][0][0] + tile_off<HD, HD, true>(row, ch);
        if (row < n && in_bounds(a.status, tp + row < a.cap))
          cp_async16(dst, (kv ? vc : kc) + (size_t)(tp + row) * HD + 8 * ch);
        else *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  };
  // int8: after the block's copies have landed, every lane reads its chunks
  // of codes, then (after __syncwarp) writes them back as fp16 over the
  // whole rows; rows past n become zero (codes and scales)
  auto widen = [&](int n) {
    if constexpr (KV8) {
      constexpr int C8 = HD / 16, L8 = C8 == 4 ? 2 : 3, MAXC = 2 * 16 * C8 / 32;
      uint4 c[MAXC];
#pragma unroll
      for (int j = 0; j < MAXC; ++j) {
        const int idx = lane + 32 * j, kv = idx >= 16 * C8, r = idx - kv * 16 * C8, row = r >> L8,
                  ch = r & (C8 - 1);
        c[j] = row < n ? reinterpret_cast<const uint4*>(&(kv ? sa.vt : sa.kt)[warp][row][0])[ch]
                       : make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
#pragma unroll
      for (int j = 0; j < MAXC; ++j) {
        const int idx = lane + 32 * j, kv = idx >= 16 * C8, r = idx - kv * 16 * C8, row = r >> L8,
                  ch = r & (C8 - 1);
        const uint32_t w[4] = {c[j].x, c[j].y, c[j].z, c[j].w};
        uint32_t h[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          h[2 * q] = pack_f16x2((float)(int8_t)(w[q] & 0xFF), (float)(int8_t)((w[q] >> 8) & 0xFF));
          h[2 * q + 1] = pack_f16x2((float)(int8_t)((w[q] >> 16) & 0xFF), (float)(int8_t)(w[q] >> 24));
        }
        uint16_t* tile = &(kv ? sa.vt : sa.kt)[warp][0][0];
        *reinterpret_cast<uint4*>(tile + tile_off<HD, HD, true>(row, 2 * ch)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(tile + tile_off<HD, HD, true>(row, 2 * ch + 1)) =
            make_uint4(h[4], h[5], h[6], h[7]);
      }
      const int kv = lane >> 4, row = lane & 15;
      if (row >= n)
#pragma unroll
        for (int k = 0; k < NG; ++k) (kv ? sa.vsc : sa.ksc)[warp][row][k] = 0;
    }
  };
  if (attend && t0 + 16 * warp < t1) stage(t0 + 16 * warp);  // each warp's first block, during the prologue
  // q heads, k, v of this kv head; RoPE factors and q/k norm weights
  for (int i = tid; i < (GQ + 2) * HD; i += NT) {
    const int r = i / HD, d = i % HD;
    const int row = r < GQ ? (g * GQ + r) * HD + d : (r == GQ ? a.q_dim + g * HD + d : a.q_dim + a.kv_dim + g * HD + d);
    sa.cur[r][d] = __ldcg(qkv + row);
  }
  const int nrope = (GQ + 1) * (HD / 2);
  // q/k norm weights: warp w takes head w (and w + 8; head GQ is k)
  float wn[2][DPL];
#pragma unroll
  for (int k2 = 0; k2 < 2; ++k2)
#pragma unroll
    for (int e = 0; e < DPL; ++e) {
      const int h = warp + 8 * k2;
      wn[k2][e] = (a.q_norm && h <= GQ) ? __ldg((h < GQ ? a.q_norm : a.k_norm) + lane + 32 * e) : 1.f;
    }
  __syncthreads();
  if (a.q_norm) {  // per-head RMSNorm of the q heads and k
#pragma unroll
    for (int k2 = 0; k2 < 2; ++k2) {
      const int h = warp + 8 * k2;
      if (h <= GQ) {
        float* v = sa.cur[h];
        float x[DPL], ss = 0.f;
#pragma unroll
        for (int e = 0; e < DPL; ++e) {
          x[e] = v[lane + 32 * e];
          ss += x[e] * x[e];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float inv = 1.0f / sqrtf(ss / (float)HD + a.eps);
#pragma unroll
        for (int e = 0; e < DPL; ++e) v[lane + 32 * e] = x[e] * inv * wn[k2][e];
      }
    }
    __syncthreads();
  }
  // RoPE of q and k; q scaled by log2(e)/sqrt(hd); k, v rounded to bf16 (the
  // last split appends them to the cache)
  const float qscale = 1.4426950408889634f / sqrtf((float)HD);
  auto keep = [&](int r, int d, float x) {
    if constexpr (KV8) {  // quantized per 32-element group below
      sa.cur[r][d] = x;
    } else {  // the warp whose block holds `pos` puts the row into its stage once its copies have landed
      const __nv_bfloat16 h = __float2bfloat16_rn(x);
      sa.cur[r][d] = __bfloat162float(h);
      if (append && in_bounds(a.status, pos < a.cap))
        (r == GQ ? kc : vc)[(size_t)pos * HD + d] = __bfloat16_as_ushort(h);
    }
  };
  for (int j = tid; j < nrope + HD; j += NT) {  // RoPE pairs of the q heads and k, then v elements
    if (j < nrope) {
      const int h = j / (HD / 2), i = j % (HD / 2);
      const float2 rcs = __ldg(a.rope + (size_t)pos * (HD / 2) + i);
      float* v = sa.cur[h];
      const int ia = a.rope_neox ? i : 2 * i, ib = a.rope_neox ? i + HD / 2 : 2 * i + 1;
      const float x0 = v[ia], x1 = v[ib];
      const float y0 = x0 * rcs.x - x1 * rcs.y, y1 = x0 * rcs.y + x1 * rcs.x;
      if (h < GQ) {
        v[ia] = y0 * qscale;
        v[ib] = y1 * qscale;
      } else {
        keep(GQ, ia, y0);
        keep(GQ, ib, y1);
      }
    } else {
      keep(GQ + 1, j - nrope, sa.cur[GQ + 1][j - nrope]);
    }
  }
  if constexpr (KV8) {
    // the grouped int8 append: warp (kv, group) quantizes 32 elements of k or
    // v (fp16 scale fp16(amax / 127), codes round(x / scale) half away from
    // zero, clamped to +-127, all in fp32); cur keeps the codes, cursc the scales
    __syncthreads();
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
      if (append && in_bounds(a.status, pos < a.cap)) {
        (kv ? vc8 : kc8)[(size_t)pos * HD + d] = (int8_t)(int)cf;
        if (lane == 0) (kv ? vs8 : ks8)[(size_t)pos * NG + grp] = __half_as_ushort(dh);
      }
    }
  }
  if (!attend) return;  // the rows' k, v are in the cache
  float* gpart = a.part + (size_t)b * bp.part_stride + (((size_t)g * a.P + split) * GQ) * (HD + 2);
  {
    // ---- warp w: blocks w, w + NW, ... of the split, each folded into the
    // warp's running (max, sum) per head and its share of o: lane holds
    // elements lane + 32e of the [GQ][HD] output
    constexpr int OE = GQ * HD / 32;
    static_assert(GQ * HD % 32 == 0, "output elements per lane");
    // the query's A fragments, packed once over the query rows of cur (the
    // same bytes: GQ * HD / 4 entries of 16 B): bf16 pairs for the bf16
    // cache's bf16 MMAs, fp16 pairs for the widened int8 codes
    constexpr int NF = GQ * HD / 4;
    static_assert(NF <= NT, "one fragment entry per thread");
    __syncthreads();  // q, k, v of this step (cur) are complete
    const uint4 qv = tid < NF ? attn_q_pack<GQ, HD, !KV8>(&sa.cur[0][0], tid) : make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    if (tid < NF) reinterpret_cast<uint4*>(&sa.cur[0][0])[tid] = qv;
    __syncthreads();
    const uint4* qp = reinterpret_cast<const uint4*>(&sa.cur[0][0]);
    float* wt = &sa.tres[warp][0][0];
    float m_run[GQ], l_run[GQ], o_run[OE];
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
      m_run[h] = -INFINITY;
      l_run[h] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < OE; ++e) o_run[e] = 0.f;
    for (int tp = t0 + 16 * warp; tp < t1; tp += 16 * NW) {
      const int n = min(16, t1 - tp);
      cp_async_wait_all();
      __syncwarp();
      widen(n);
      __syncwarp();
      if (pos >= tp && pos < tp + n) {  // this step's k, v row (its copy from the cache may predate the append)
        for (int i = lane; i < 2 * HD; i += 32) {
          const int kv = i >= HD, d = i - kv * HD;
          // bf16: the bf16-exact value; int8: its code, exactly in fp16
          const uint16_t v = KV8 ? __half_as_ushort(__float2half_rn(sa.cur[GQ + kv][d]))
                                 : (uint16_t)(__float_as_uint(sa.cur[GQ + kv][d]) >> 16);
          (kv ? &sa.vt[warp][0][0] : &sa.kt[warp][0][0])[tile_off<HD, HD, true>(pos - tp, d >> 3) + (d & 7)] = v;
        }
        if constexpr (KV8)
          if (lane < 2 * NG)
            (lane < NG ? sa.ksc : sa.vsc)[warp][pos - tp][lane % NG] =
                __half_as_ushort(__float2half_rn(sa.cursc[lane / NG][lane % NG]));
        __syncwarp();
      }
      if constexpr (KV8)
        attn_block16_q8<GQ, HD, HD, true>(reinterpret_cast<const float*>(qp), &sa.kt[warp][0][0], &sa.vt[warp][0][0],
                                          &sa.ksc[warp][0][0], &sa.vsc[warp][0][0], 0, n, lane, wt, HD + 2);
      else
        attn_block16_bf<GQ, HD>(qp, &sa.kt[warp][0][0], &sa.vt[warp][0][0], n, lane, wt, HD + 2);
      __syncwarp();  // the stage has been read and the block's results written
      if (tp + 16 * NW < t1) stage(tp + 16 * NW);
      float fr[GQ], fb[GQ];
#pragma unroll
      for (int h = 0; h < GQ; ++h) {
        const float mb = wt[h * (HD + 2) + HD], lb = wt[h * (HD + 2) + HD + 1];
        const float M = fmaxf(m_run[h], mb);
        fr[h] = m_run[h] == -INFINITY ? 0.f : exp2f(m_run[h] - M);
        fb[h] = exp2f(mb - M);
        l_run[h] = l_run[h] * fr[h] + lb * fb[h];
        m_run[h] = M;
      }
#pragma unroll
      for (int e = 0; e < OE; ++e) {
        const int i = lane + 32 * e, h = i / HD, d = i % HD;
        o_run[e] = o_run[e] * fr[h] + wt[h * (HD + 2) + d] * fb[h];
      }
      __syncwarp();  // the next block's results overwrite wt
    }
    // the warps' states -> tres, then the split's partial (warps in order)
#pragma unroll
    for (int e = 0; e < OE; ++e) {
      const int i = lane + 32 * e;
      wt[(i / HD) * (HD + 2) + i % HD] = o_run[e];
    }
    if (lane < GQ) {
#pragma unroll
      for (int h = 0; h < GQ; ++h)
        if (h == lane) {
          wt[h * (HD + 2) + HD] = m_run[h];
          wt[h * (HD + 2) + HD + 1] = l_run[h];
        }
    }
    __syncthreads();
    for (int i = tid; i < GQ * HD; i += NT) {
      const int h = i / HD, d = i % HD;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NW; ++w) M = fmaxf(M, sa.tres[w][h][HD]);
      float O = 0.f, L = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float mw = sa.tres[w][h][HD];
        const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);
        O += sa.tres[w][h][d] * f;
        L += sa.tres[w][h][HD + 1] * f;
      }
      gpart[h * (HD + 2) + d] = O;
      if (d == 0) {
        gpart[h * (HD + 2) + HD] = M;
        gpart[h * (HD + 2) + HD + 1] = L;
      }
    }
  }
  // ---- the last split of this (sequence, kv head) merges the splits (no waiting)
  int* counter = a.counter + (size_t)b * a.Hkv + g;
  __threadfence();
  __syncthreads();
  if (tid == 0) sa.is_last = (atomicAdd(counter, 1) == P_eff - 1);
  __syncthreads();
  if (!sa.is_last) return;
  __threadfence();
  // the last split: (max, sum) of every split and head to shared memory while
  // each thread loads its output element of every split (one round trip)
  const float* hp = a.part + (size_t)b * bp.part_stride + ((size_t)g * a.P * GQ) * (HD + 2);
  float* ml = &sa.tres[0][0][0];  // [P_eff][GQ][2] (the block results are no longer needed)
  static_assert(sizeof(sa.tres) >= PMAX * GQ * 2 * sizeof(float), "merge scratch");
  for (int i = tid; i < P_eff * GQ * 2; i += NT) {
    const int sidx = i / (2 * GQ), h = (i / 2) % GQ, e = i & 1;
    ml[i] = __ldcg(hp + ((size_t)sidx * GQ + h) * (HD + 2) + HD + e);
  }
  for (int i0 = 0; i0 < GQ * HD; i0 += NT) {
    const int i = i0 + tid, h = i / HD, d = i % HD;
    float ov[PMAX];
#pragma unroll
    for (int s2 = 0; s2 < PMAX; ++s2)
      ov[s2] = ldcg1_if(hp + ((size_t)s2 * GQ + (i < GQ * HD ? h : 0)) * (HD + 2) + d, s2 < P_eff && i < GQ * HD);
    __syncthreads();
    if (i < GQ * HD) {
      float M = -INFINITY;
      for (int s2 = 0; s2 < P_eff; ++s2) M = fmaxf(M, ml[(s2 * GQ + h) * 2]);
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < PMAX; ++s2)
        if (s2 < P_eff) {
          const float f = exp2f(ml[(s2 * GQ + h) * 2] - M);
          L += ml[(s2 * GQ + h) * 2 + 1] * f;
          O += ov[s2] * f;
        }
      store_hl(bp.o_hl, bp.o_cols, b, (g * GQ + h) * HD + d, O / L);
    }
  }
  if (tid == 0) *counter = 0;
}

}  // namespace llmq
