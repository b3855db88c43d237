// Warp-level flash-decoding on the tensor cores (mma.sync m16n8k16, fp16
// operands, fp32 accumulation) for the decode step.
//
// One warp scores the GQ query heads of a kv head against 16 cached
// positions and forms their softmax-weighted V sum. The cached bf16 K/V are
// staged as fp16, which holds every bf16 value of magnitude 2^-14 .. 65504
// exactly. The M = 16 rows of the A operand hold the fp16 high parts of the
// GQ heads (rows 0..GQ-1) and the fp16 remainders (rows 8..8+GQ-1), so one MMA
// computes both halves and their sum carries a 22-bit-mantissa query
// (relative error ~2^-22); the probabilities are split the same way for P V.
// K/V rows sit in shared memory with a padded row stride (RS = HD + 8
// halves), which makes the ldmatrix row fetches of a fragment hit distinct
// bank groups.
#pragma once
#include "common.cuh"

namespace llmq {

__device__ __forceinline__ uint32_t pack_f16x2(float e0, float e1) {
  const __half2 v = __floats2half2_rn(e0, e1);  // e0 in the low half
  return *reinterpret_cast<const uint32_t*>(&v);
}
// x = hi + lo with hi = fp16(x); lo is exact in fp32 (rounded to fp16 when packed)
__device__ __forceinline__ void split_f16(float x, float& hi, float& lo) {
  hi = __half2float(__float2half_rn(x));
  lo = x - hi;
}
// Two bf16 (a packed pair) -> two fp16, exact for magnitudes 2^-14 .. 65504.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float e0, float e1) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(e0, e1);  // e0 in the low half
  return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

// A fragment of the query block for dims 16ks .. 16ks+15: q is [GQ][HD] fp32
// in shared memory (already scaled). Lane (g = lane/4, t = lane%4) holds rows
// g / g+8 = fp16 high part / remainder of head g at dims 16ks+2t(+1) and +8.
template <int GQ, int HD>
__device__ __forceinline__ void attn_q_frag(uint32_t (&qf)[4], const float* q, int ks, int lane) {
  const int g = lane >> 2, t = lane & 3;
  float x[4] = {0.f, 0.f, 0.f, 0.f};
  if (g < GQ) {
    const float2 a = *reinterpret_cast<const float2*>(q + g * HD + 16 * ks + 2 * t);
    const float2 b = *reinterpret_cast<const float2*>(q + g * HD + 16 * ks + 2 * t + 8);
    x[0] = a.x;
    x[1] = a.y;
    x[2] = b.x;
    x[3] = b.y;
  }
  float h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) split_f16(x[i], h[i], l[i]);
  qf[0] = pack_f16x2(h[0], h[1]);
  qf[1] = pack_f16x2(l[0], l[1]);
  qf[2] = pack_f16x2(h[2], h[3]);
  qf[3] = pack_f16x2(l[2], l[3]);
}

// Offset (in halves) of dims 8c .. 8c+7 of row r of a K/V tile. Padded tiles
// (SWZ = false): rows of RS > HD halves. Unpadded tiles (SWZ = true, rows of
// HD halves): chunk c of row r sits at chunk c ^ (r & 7), so the 8 rows of an
// ldmatrix fetch still hit distinct bank groups.
template <int HD, int RS, bool SWZ>
__device__ __forceinline__ int tile_off(int r, int c) {
  if constexpr (SWZ) return r * HD + 8 * (c ^ (r & 7));
  else return r * RS + 8 * c;
}

// The query block's A fragments, built once per attention item: entry
// ks * 4 GQ + 4 g + t holds lane (g, t)'s four registers for dims 16ks ..
// 16ks+15 (as attn_q_frag), high parts and remainders as bf16 (BF) or fp16
// pairs. Lanes with g >= GQ take zeros.
template <int GQ, int HD, bool BF>
__device__ __forceinline__ uint4 attn_q_pack(const float* q, int f) {
  const int ks = f / (4 * GQ), g = (f / 4) % GQ, t = f % 4;
  const float* r = q + g * HD + 16 * ks + 2 * t;
  const float x[4] = {r[0], r[1], r[8], r[9]};
  float h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (BF) {
      h[i] = __bfloat162float(__float2bfloat16_rn(x[i]));
      l[i] = x[i] - h[i];
    } else {
      split_f16(x[i], h[i], l[i]);
    }
  }
  if constexpr (BF)
    return make_uint4(pack_bf16x2(h[0], h[1]), pack_bf16x2(l[0], l[1]), pack_bf16x2(h[2], h[3]),
                      pack_bf16x2(l[2], l[3]));
  else
    return make_uint4(pack_f16x2(h[0], h[1]), pack_f16x2(l[0], l[1]), pack_f16x2(h[2], h[3]),
                      pack_f16x2(l[2], l[3]));
}
template <int GQ>
__device__ __forceinline__ void attn_q_load(uint32_t (&qf)[4], const uint4* qp, int ks, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const uint4 v = g < GQ ? qp[ks * 4 * GQ + 4 * g + t] : make_uint4(0u, 0u, 0u, 0u);
  qf[0] = v.x;
  qf[1] = v.y;
  qf[2] = v.z;
  qf[3] = v.w;
}

// attn_block16 on bf16 operands: the cache's bf16 K/V rows as they are
// (unpadded, tile_off's permuted chunks, rows 0..15), the query's packed bf16
// fragments (attn_q_pack), the probabilities split into bf16 high part and
// remainder (16-bit mantissa, relative error ~2^-17), fp32 accumulation.
// Same outputs as attn_block16.
template <int GQ, int HD>
__device__ __forceinline__ void attn_block16_bf(const uint4* qp, const uint16_t* kt, const uint16_t* vt, int nvalid,
                                                int lane, float* out, int OS) {
  const int g = lane >> 2, t = lane & 3, r8 = lane & 7, mi = lane >> 3;
  float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
  for (int ks = 0; ks < HD / 16; ++ks) {
    uint32_t qf[4];
    attn_q_load<GQ>(qf, qp, ks, lane);
    uint32_t b[4];
    ldsm_x4(b, kt + tile_off<HD, HD, true>(8 * (mi >> 1) + r8, 2 * ks + (mi & 1)));
    mma_bf16_16816(s[0], qf, b[0], b[1]);
    mma_bf16_16816(s[1], qf, b[2], b[3]);
  }
  float sc[4];
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int li = 8 * j + 2 * t + e;
      sc[2 * j + e] = li < nvalid ? s[j][e] + s[j][e + 2] : -INFINITY;  // high rows + remainder rows
    }
  float mx = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  float p[4], sum = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    p[i] = exp2f(sc[i] - mx);
    sum += p[i];
  }
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  float ph[4], pl[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    ph[i] = __bfloat162float(__float2bfloat16_rn(p[i]));
    pl[i] = p[i] - ph[i];
  }
  const uint32_t pa[4] = {pack_bf16x2(ph[0], ph[1]), pack_bf16x2(pl[0], pl[1]), pack_bf16x2(ph[2], ph[3]),
                          pack_bf16x2(pl[2], pl[3])};
  float* o = out + g * OS;
  const bool mine = g < GQ;
#pragma unroll
  for (int nt = 0; nt < HD / 8; nt += 2) {
    uint32_t b[4];
    ldsm_x4_t(b, vt + tile_off<HD, HD, true>(8 * (mi & 1) + r8, nt + (mi >> 1)));
    float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
    mma_bf16_16816(d0, pa, b[0], b[1]);
    mma_bf16_16816(d1, pa, b[2], b[3]);
    if (mine) {
      *reinterpret_cast<float2*>(o + 8 * nt + 2 * t) = make_float2(d0[0] + d0[2], d0[1] + d0[3]);
      *reinterpret_cast<float2*>(o + 8 * nt + 8 + 2 * t) = make_float2(d1[0] + d1[2], d1[1] + d1[3]);
    }
  }
  if (mine && t == 0) {
    o[HD] = mx;
    o[HD + 1] = sum;
  }
}

// One warp, the GQ heads of q ([GQ][HD], scaled) against the 16 staged rows
// row0 .. row0+15 (rows at or beyond `nvalid` are zero-filled and masked).
// Scores are in the log2 domain (q carries log2(e)/sqrt(hd)). Lane (head
// g = lane/4 < GQ, t = lane%4) writes to out[g*OS ..]: o at dims 8nt+2t(+1)
// (sum over the 16 positions of 2^(s - m) v), and lane t = 0 writes m (max
// score) at [HD] and l (sum of 2^(s - m)) at [HD+1].
template <int GQ, int HD, int RS>
__device__ __forceinline__ void attn_block16(const float* q, const uint16_t* kt, const uint16_t* vt, int row0,
                                             int nvalid, int lane, float* out, int OS) {
  const int g = lane >> 2, t = lane & 3, r8 = lane & 7, mi = lane >> 3;
  float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
  for (int ks = 0; ks < HD / 16; ++ks) {
    uint32_t qf[4];
    attn_q_frag<GQ, HD>(qf, q, ks, lane);
    // matrices: positions 0-7 / 8-15 (n-tile j = mi/2) x dims 16ks + 8*(mi%2) .. +7
    uint32_t b[4];
    ldsm_x4(b, kt + (size_t)(row0 + 8 * (mi >> 1) + r8) * RS + 16 * ks + 8 * (mi & 1));
    mma_f16_16816(s[0], qf, b[0], b[1]);
    mma_f16_16816(s[1], qf, b[2], b[3]);
  }
  float sc[4];
#pragma unroll
  for (int j = 0; j < 2; ++j)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int li = 8 * j + 2 * t + e;
      sc[2 * j + e] = li < nvalid ? s[j][e] + s[j][e + 2] : -INFINITY;  // high rows + remainder rows
    }
  float mx = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  float p[4], sum = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    p[i] = exp2f(sc[i] - mx);
    sum += p[i];
  }
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  float ph[4], pl[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) split_f16(p[i], ph[i], pl[i]);
  const uint32_t pa[4] = {pack_f16x2(ph[0], ph[1]), pack_f16x2(pl[0], pl[1]), pack_f16x2(ph[2], ph[3]),
                          pack_f16x2(pl[2], pl[3])};
  float* o = out + g * OS;
  const bool mine = g < GQ;
#pragma unroll
  for (int nt = 0; nt < HD / 8; nt += 2) {
    // matrices (transposed): positions 8*(mi%2) .. +7 x dims 8*(nt + mi/2) .. +7
    uint32_t b[4];
    ldsm_x4_t(b, vt + (size_t)(row0 + 8 * (mi & 1) + r8) * RS + 8 * (nt + (mi >> 1)));
    float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
    mma_f16_16816(d0, pa, b[0], b[1]);
    mma_f16_16816(d1, pa, b[2], b[3]);
    if (mine) {
      *reinterpret_cast<float2*>(o + 8 * nt + 2 * t) = make_float2(d0[0] + d0[2], d0[1] + d0[3]);
      *reinterpret_cast<float2*>(o + 8 * nt + 8 + 2 * t) = make_float2(d1[0] + d1[2], d1[1] + d1[3]);
    }
  }
  if (mine && t == 0) {
    o[HD] = mx;
    o[HD + 1] = sum;
  }
}

// attn_block16 on the CUDA cores (fp32 FMAs on the staged fp16 rows), the
// same inputs and outputs: the comparison the tensor-core block is measured
// against (step kernels built with LLMQ_ATTN_CUDA_CORES=1). Lane (position
// p = lane % 16, head parity lane / 16) scores its position against heads
// lane/16, lane/16 + 2, ...; the softmax of a head reduces over 16 lanes;
// then lane d accumulates output dims d, d + 32, ... of every head, taking
// each position's probability by a shuffle.
template <int GQ, int HD, int RS>
__device__ __forceinline__ void attn_block16_cc(const float* q, const uint16_t* kt, const uint16_t* vt, int row0,
                                                int nvalid, int lane, float* out, int OS) {
  constexpr int NH = (GQ + 1) / 2;  // heads per lane
  const int p = lane & 15, hp = lane >> 4;
  float sc[NH];
  const __half2* kr = reinterpret_cast<const __half2*>(kt + (size_t)(row0 + p) * RS);
#pragma unroll
  for (int j = 0; j < NH; ++j) sc[j] = 0.f;
#pragma unroll 8
  for (int d2 = 0; d2 < HD / 2; ++d2) {
    const float2 k = __half22float2(kr[d2]);
#pragma unroll
    for (int j = 0; j < NH; ++j) {
      const int h = hp + 2 * j;
      if (h < GQ) {
        const float2 qq = *reinterpret_cast<const float2*>(q + h * HD + 2 * d2);
        sc[j] = fmaf(qq.x, k.x, fmaf(qq.y, k.y, sc[j]));
      }
    }
  }
  float pr[NH], mx[NH], sm[NH];
#pragma unroll
  for (int j = 0; j < NH; ++j) {
    const float v = p < nvalid ? sc[j] : -INFINITY;
    float m = v;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    pr[j] = exp2f(v - m);
    float l = pr[j];
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    mx[j] = m;
    sm[j] = l;
  }
  float acc[GQ][HD / 32];
#pragma unroll
  for (int h = 0; h < GQ; ++h)
#pragma unroll
    for (int e = 0; e < HD / 32; ++e) acc[h][e] = 0.f;
#pragma unroll 4
  for (int pp = 0; pp < 16; ++pp) {
    float v[HD / 32];
#pragma unroll
    for (int e = 0; e < HD / 32; ++e)
      v[e] = __half2float(__ushort_as_half(vt[(size_t)(row0 + pp) * RS + lane + 32 * e]));
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
      const float w = __shfl_sync(0xffffffffu, pr[h / 2], pp + 16 * (h & 1));
#pragma unroll
      for (int e = 0; e < HD / 32; ++e) acc[h][e] = fmaf(w, v[e], acc[h][e]);
    }
  }
#pragma unroll
  for (int h = 0; h < GQ; ++h)
#pragma unroll
    for (int e = 0; e < HD / 32; ++e) out[h * OS + lane + 32 * e] = acc[h][e];
  if (p == 0)
#pragma unroll
    for (int j = 0; j < NH; ++j)
      if (hp + 2 * j < GQ) {
        out[(hp + 2 * j) * OS + HD] = mx[j];
        out[(hp + 2 * j) * OS + HD + 1] = sm[j];
      }
}

// attn_block16 over int8 K/V (the grouped int8 cache): kt/vt hold the codes
// as fp16 (exact), ks/vs the staged rows' fp16 group scales [row][HD / 32].
// A key group's scale multiplies that group's partial scores per position
// (the MMAs of a group's two 16-dim slices accumulate apart). A value
// group's scale folds into the probabilities before P V; dividing it by the
// block's largest scale of the group keeps the scaled probabilities in [0, 1]
// for their fp16 high/low split, and that largest scale multiplies the MMA
// result back. Same outputs as attn_block16. SWZ: unpadded fp16 rows with
// tile_off's permuted chunks instead of padded rows, and q holds the packed
// fp16 fragments (attn_q_pack) instead of the query.
template <int GQ, int HD, int RS, bool SWZ = false>
__device__ __forceinline__ void attn_block16_q8(const float* q, const uint16_t* kt, const uint16_t* vt,
                                                const uint16_t* ks, const uint16_t* vs, int row0, int nvalid,
                                                int lane, float* out, int OS) {
  constexpr int NG = HD / 32;
  const int g = lane >> 2, t = lane & 3, r8 = lane & 7, mi = lane >> 3;
  float s[NG][2][4];
#pragma unroll
  for (int k = 0; k < NG; ++k)
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[k][j][e] = 0.f;
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    uint32_t qf[4];
    if constexpr (SWZ) attn_q_load<GQ>(qf, reinterpret_cast<const uint4*>(q), kk, lane);
    else attn_q_frag<GQ, HD>(qf, q, kk, lane);
    uint32_t b[4];
    ldsm_x4(b, kt + tile_off<HD, RS, SWZ>(row0 + 8 * (mi >> 1) + r8, 2 * kk + (mi & 1)));
    mma_f16_16816(s[kk / 2][0], qf, b[0], b[1]);
    mma_f16_16816(s[kk / 2][1], qf, b[2], b[3]);
  }
  // this lane's positions: 2t, 2t+1, 2t+8, 2t+9 of the block (score / probability i)
  int li[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) li[i] = 8 * (i >> 1) + 2 * t + (i & 1);
  float sc[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int j = i >> 1, e = i & 1;
    float v = 0.f;
#pragma unroll
    for (int k = 0; k < NG; ++k)
      v += __half2float(__ushort_as_half(ks[(row0 + li[i]) * NG + k])) * (s[k][j][e] + s[k][j][e + 2]);
    sc[i] = li[i] < nvalid ? v : -INFINITY;
  }
  float mx = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  float p[4], sum = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    p[i] = exp2f(sc[i] - mx);
    sum += p[i];
  }
  sum += __shfl_xor_sync(0xffffffffu, sum, 1);
  sum += __shfl_xor_sync(0xffffffffu, sum, 2);
  float* o = out + g * OS;
  const bool mine = g < GQ;
#pragma unroll
  for (int vg = 0; vg < NG; ++vg) {
    float r[4], smax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      r[i] = __half2float(__ushort_as_half(vs[(row0 + li[i]) * NG + vg]));
      smax = fmaxf(smax, r[i]);
    }
    smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, 1));
    smax = fmaxf(smax, __shfl_xor_sync(0xffffffffu, smax, 2));
    const float inv = smax > 0.f ? 1.0f / smax : 0.f;
    float ph[4], pl[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) split_f16(p[i] * (r[i] * inv), ph[i], pl[i]);
    const uint32_t pa[4] = {pack_f16x2(ph[0], ph[1]), pack_f16x2(pl[0], pl[1]), pack_f16x2(ph[2], ph[3]),
                            pack_f16x2(pl[2], pl[3])};
#pragma unroll
    for (int nt = 4 * vg; nt < 4 * vg + 4; nt += 2) {
      uint32_t b[4];
      ldsm_x4_t(b, vt + tile_off<HD, RS, SWZ>(row0 + 8 * (mi & 1) + r8, nt + (mi >> 1)));
      float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
      mma_f16_16816(d0, pa, b[0], b[1]);
      mma_f16_16816(d1, pa, b[2], b[3]);
      if (mine) {
        *reinterpret_cast<float2*>(o + 8 * nt + 2 * t) = make_float2((d0[0] + d0[2]) * smax, (d0[1] + d0[3]) * smax);
        *reinterpret_cast<float2*>(o + 8 * nt + 8 + 2 * t) =
            make_float2((d1[0] + d1[2]) * smax, (d1[1] + d1[3]) * smax);
      }
    }
  }
  if (mine && t == 0) {
    o[HD] = mx;
    o[HD + 1] = sum;
  }
}

}  // namespace llmq
