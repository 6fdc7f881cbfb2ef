// Decode attention over a ROCmFP4 K/V cache (one query token per sequence):
//   out[b][h] = softmax_t(scale * q[b][h] . K[b][hk][t]) . V[b][hk][t],  t < lens[b],
// with hk = h / (H / Hkv), fp32 output.  K and V rows (one per token and KV
// head) are ROCmFP4 blocks along the head dimension D, and are decoded in
// registers: no dequantised copy of the cache is ever written.  This is the
// reading of the "FlashAttention K/V cache optimization" item of
// "Feasibility Report: Porting ROCmFP4 to Atlas" (sections "Why AMD is
// Different from NVIDIA" and "Option 2"); the block decode follows section
// "What is ROCmFP4?" (Block Layout, Codebook10 Value Table, Scale Format).
//
// Split kernel.  A CTA takes one (sequence, KV head) and a contiguous range of
// its 32-token chunks (a flash-decoding split); its 4 warps take alternate
// chunks, each staging the chunk's K and V rows with bulk copies into a ring
// of its own and keeping an online softmax for the G = H / Hkv query heads of
// the group (G <= 8):
//   scores: mma.sync m16n8k16, A = 16 tokens x 16 of D (decoded K, exact in
//           fp16 / bf16), B = the G heads' q (the MMA's 8 columns);
//   softmax in fp32, base 2 (scores pre-multiplied by scale * log2 e);
//   P.V:    mma.sync with A = 16 of D x 16 tokens of V^T (decoded V rows
//           transposed in registers by movmatrix) and B = P^T.  P is split
//           into an fp16 high part and an fp16 remainder (scaled by 2^15
//           into fp16's normal range), so the products keep fp32 precision.
// The warps' states are merged in shared memory in warp order.  With one
// split the CTA writes the output; otherwise it writes its unnormalised
// partial (max, sum, P.V) and the combine kernel merges the splits in split
// order.  Every order is fixed, so results are bitwise repeatable.
//
// Byte order inside a block (read as in ggml Q4_0): byte j holds weight j (low nibble) and
// weight j+16 (high nibble), so cvt.rn.f16x2.e2m1x2 of byte j gives the pair
// (d = j, d = j + 16) of that block.  Lane (r, c) = (lane / 4, lane % 4)
// decodes bytes 4c .. 4c+3 of every block of its tokens; the MMA k order is
// chosen to match (B fragments of q and of P follow the same order).
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace rocmfp4 {
namespace {

constexpr int kAttnWarps = 4;
constexpr int kChunk = 32;      // tokens per warp step
constexpr int kAttnStages = 2;  // ring depth per warp
constexpr float kPScale = 32768.0f;
constexpr float kPUnscale = 1.0f / 32768.0f;
constexpr float kLog2e = 1.4426950408889634f;

struct AttnParams {
  const uint16_t* q;  // [B][H][D] fp16 / bf16 bits
  const uint8_t* K;   // [B][Hkv][Tmax] rows of D/32 blocks
  const uint8_t* V;
  const int32_t* lens;  // [B]
  float* out;           // [B][H][D]
  float* ws;            // split partials, attn_partial_floats(D) each
  int B, H, Hkv, G, Tmax, S;
  float scale_log2;  // softmax scale * log2(e)
  uint32_t* err;
};

RF4_HOSTDEV constexpr int partial_floats(int D) { return 16 + 8 * D; }

template <int V, int D>
struct AttnFmt {
  static constexpr int BB = Fmt<V>::BB;             // block bytes
  static constexpr int NB = D / 32;                 // blocks per row
  static constexpr int RB = NB * BB;                // row bytes
  static constexpr int CB = kChunk * RB;            // chunk bytes (K or V)
  static constexpr int STAGE = 2 * CB;              // K chunk then V chunk
  static constexpr int KS = D / 16;                 // MMA k steps over D
  static constexpr int WARP_RING = kAttnStages * STAGE;
  static constexpr int MERGE = partial_floats(D) * 4;  // one warp's state for the merge
  // per warp: its ring; the merge area reuses the rings
  static constexpr int WARP_BYTES = WARP_RING;
  static constexpr int BAR_OFF = kAttnWarps * WARP_BYTES;
  static constexpr int SMEM = BAR_OFF + kAttnWarps * kAttnStages * 8;
  static_assert(kAttnWarps * MERGE <= kAttnWarps * WARP_RING, "merge area fits in the rings");
  static_assert(CB % 16 == 0, "bulk copies of whole chunks");
};

// Shared-memory loads are plain C++ loads, so the compiler may schedule them
// early (the mbarrier wait and the proxy fence carry "memory" clobbers, which
// keep them after the data lands and before the stage is refilled).
RF4_DEV uint32_t lds32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

// Four bytes at any shared-memory address (two aligned words and a funnel shift).
RF4_DEV uint32_t lds_bytes4(const uint8_t* p) {
  const uint32_t mis = (uint32_t)reinterpret_cast<uintptr_t>(p) & 3u;
  const uint8_t* a = p - mis;
  return __funnelshift_r(lds32(a), lds32(a + 4), mis * 8u);
}

// Four bytes at an address whose offset from a 4-byte boundary is al (0..3),
// or not known (al = -1).  Called with al a constant after unrolling, so the
// branches fold away.
RF4_DEV uint32_t lds_bytes4_al(const uint8_t* p, int al) {
  if (al == 0) return lds32(p);
  if (al > 0) return __funnelshift_r(lds32(p - al), lds32(p - al + 4), 8 * al);
  return lds_bytes4(p);
}

// Offset from a 4-byte boundary of byte `off` of a token row, when rows start
// on 4-byte boundaries (every row length here is a multiple of 4 except the
// single-scale rows of D = 64), else -1.
template <int V, int D>
RF4_HOSTDEV constexpr int row_align(int off) {
  return (Fmt<V>::BB * (D / 32)) % 4 == 0 ? off % 4 : -1;
}

// Scale pair of a block as f16x2 E4M3 values: (scale of weights 0-15, scale
// of weights 16-31); the single-scale variant repeats its one scale.
template <int V>
RF4_DEV uint32_t block_scales(const uint8_t* block, int al) {
  const uint8_t* a = block + 16;
  const uint32_t mis = (uint32_t)reinterpret_cast<uintptr_t>(a) & 3u;
  const uint32_t w = al >= 0 ? lds32(a - al) >> (8 * al) : lds32(a - mis) >> (mis * 8u);
  if constexpr (V == 0) {
    return e4m3x2<0>(w & 0xFFFFu);  // two bytes, never straddling a word (even address)
  } else {
    return e4m3x2<0>(__byte_perm(w, 0u, 0x0000u) & 0xFFFFu);  // the byte twice
  }
}

// The four decoded pairs of bytes 4c .. 4c+3 of a block, each
// (w_j, w_{j+16}) * (scale pair), exact in fp16.
RF4_DEV void decode4(uint32_t codes, uint32_t s2, uint32_t (&v)[4]) {
  v[0] = hmul2(clamp5(e2m1x2<0>(codes)), s2);
  v[1] = hmul2(clamp5(e2m1x2<1>(codes)), s2);
  v[2] = hmul2(clamp5(e2m1x2<2>(codes)), s2);
  v[3] = hmul2(clamp5(e2m1x2<3>(codes)), s2);
}

// The MMA and movmatrix wrappers below touch registers only, so they are not
// volatile: the compiler may schedule them among the softmax's dependent steps.
RF4_DEV void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

RF4_DEV void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 8 x 8 transpose of 16-bit elements across the warp (fragment layout: lane
// (r, c) holds elements (r, 2c) and (r, 2c+1)).
RF4_DEV uint32_t movmatrix_t(uint32_t a) {
  uint32_t d;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// 2^x by the hardware approximation (relative error about 2^-22; 2^-inf = +0,
// subnormal results flush to zero).
RF4_DEV float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

RF4_DEV uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// p = hi + lo in two fp16 pairs (p already scaled by 2^15).
// C = 0 form of mma_f16 / mma_bf16.
RF4_DEV void mma_z(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1, bool bf16) {
  const float z = 0.f;
  if (bf16)
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
  else
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(z));
}

RF4_DEV void split_half2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = pack_half2(a - __low2float(h), b - __high2float(h));
}

template <int V, int ACT, int D>
__global__ void __launch_bounds__(kAttnWarps * 32) attn_split_kernel(const __grid_constant__ AttnParams p) {
  using F = AttnFmt<V, D>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, c = lane & 3;  // fragment row (token / head) and column group
  const int S = p.S, G = p.G;
  const int bhk = blockIdx.x / S, split = blockIdx.x % S;
  const int b = bhk / p.Hkv, hk = bhk % p.Hkv;
  uint8_t* ring = smem + (size_t)warp * F::WARP_BYTES;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + F::BAR_OFF) + warp * kAttnStages;
  if (lane == 0) {
    for (int i = 0; i < kAttnStages; ++i) mbar_init(smem_addr(&bars[i]), 1);
    fence_mbar_init();
  }
  __syncwarp();
  // Everything read below may be written by the preceding kernel on the stream.
  grid_dependency_wait();

  int T = p.lens[b];
  T = T < 0 ? 0 : (T > p.Tmax ? p.Tmax : T);
  const int nch = (T + kChunk - 1) / kChunk;
  const int c0 = (int)((int64_t)split * nch / S), c1 = (int)((int64_t)(split + 1) * nch / S);
  const uint8_t* Kb = p.K + (size_t)bhk * p.Tmax * F::RB;
  const uint8_t* Vb = p.V + (size_t)bhk * p.Tmax * F::RB;

  // B fragments of q: k step (block kb, half h) pairs byte j = 4c + 2h of
  // every block with column (2c, 2c+1) and byte j + 1 with (2c+8, 2c+9).
  uint32_t qb0[F::KS], qb1[F::KS];
  {
    const int g = r;  // B column = query head of the group
    const uint16_t* qr = p.q + ((size_t)b * p.H + (size_t)hk * G + (g < G ? g : 0)) * D;
#pragma unroll
    for (int ks = 0; ks < F::KS; ++ks) {
      const int kb = ks / 2, h = ks % 2;
      const int d0 = 32 * kb + 4 * c + 2 * h;
      const uint32_t x0 = qr[d0], x16 = qr[d0 + 16], x1 = qr[d0 + 1], x17 = qr[d0 + 17];
      qb0[ks] = g < G ? (x0 | (x16 << 16)) : 0u;
      qb1[ks] = g < G ? (x1 | (x17 << 16)) : 0u;
    }
  }

  // online softmax state of heads 2c and 2c+1 (base-2 scores), and P.V in
  // fragments: oacc[m] for D rows 16m .. 16m+15 (block m/2, half m%2)
  // (lrun holds this lane's tokens only; the lanes' parts are added after the loop)
  float mrun[2] = {-INFINITY, -INFINITY}, lrun[2] = {0.f, 0.f};
  float oacc[2 * F::NB][4];
#pragma unroll
  for (int m = 0; m < 2 * F::NB; ++m) oacc[m][0] = oacc[m][1] = oacc[m][2] = oacc[m][3] = 0.f;

  auto issue = [&](int ch, int st) {
    if (lane == 0) {
      const uint32_t bar = smem_addr(&bars[st]);
      mbar_arrive_expect_tx(bar, (uint32_t)F::STAGE);
      uint8_t* dst = ring + (size_t)st * F::STAGE;
      bulk_g2s(smem_addr(dst), Kb + (size_t)ch * F::CB, F::CB, bar);
      bulk_g2s(smem_addr(dst + F::CB), Vb + (size_t)ch * F::CB, F::CB, bar);
    }
  };
  int issued = 0, n_mine = 0;
  for (int ch = c0 + warp; ch < c1; ch += kAttnWarps) ++n_mine;
  for (; issued < kAttnStages && issued < n_mine; ++issued) issue(c0 + warp + issued * kAttnWarps, issued);

  bool ok = true;
  for (int i = 0; i < n_mine && ok; ++i) {
    const int ch = c0 + warp + i * kAttnWarps;
    const int st = i % kAttnStages;
    if (!mbar_wait_bounded(smem_addr(&bars[st]), (uint32_t)((i / kAttnStages) & 1))) {
      ok = false;
      break;
    }
    const uint8_t* ks_base = ring + (size_t)st * F::STAGE;
    const uint8_t* vs_base = ks_base + F::CB;
    const int t0 = ch * kChunk;  // first token of the chunk

    // ---- scores: token rows 16mt + r and 16mt + r + 8 ----
    float sacc[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const uint8_t* ra = ks_base + (16 * mt + r) * F::RB;
      const uint8_t* rb = ra + 8 * F::RB;
#pragma unroll
      for (int kb = 0; kb < F::NB; ++kb) {
        uint32_t va[4], vb[4];
        const int alc = row_align<V, D>(kb * F::BB), als = row_align<V, D>(kb * F::BB + 16);
        decode4(lds_bytes4_al(ra + kb * F::BB + 4 * c, alc), block_scales<V>(ra + kb * F::BB, als), va);
        decode4(lds_bytes4_al(rb + kb * F::BB + 4 * c, alc), block_scales<V>(rb + kb * F::BB, als), vb);
        if constexpr (ACT == 1) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            va[k] = f16x2_to_bf16x2(va[k]);
            vb[k] = f16x2_to_bf16x2(vb[k]);
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t a[4] = {va[2 * h], vb[2 * h], va[2 * h + 1], vb[2 * h + 1]};
          if (kb == 0 && h == 0)  // the first step starts from zero
            mma_z(sacc[mt], a, qb0[0], qb1[0], ACT == 1);
          else if constexpr (ACT == 1)
            mma_bf16(sacc[mt], a, qb0[2 * kb + h], qb1[2 * kb + h]);
          else
            mma_f16(sacc[mt], a, qb0[2 * kb + h], qb1[2 * kb + h]);
        }
      }
    }

    // ---- online softmax over the chunk (heads 2c, 2c+1 in this lane) ----
    // Every chunk holds at least one token of the sequence, so each running
    // max is finite from the first chunk on, and 2^(-inf - max) = 0 needs no
    // guard.
    float x[2][4], cmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) x[mt][e] = sacc[mt][e] * p.scale_log2;
    if (t0 + kChunk > T) {  // only the last chunk has tokens past the sequence
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (t0 + 16 * mt + r + (e >= 2 ? 8 : 0) >= T) x[mt][e] = -INFINITY;
    }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) cmax[e & 1] = fmaxf(cmax[e & 1], x[mt][e]);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      cmax[j] = fmaxf(cmax[j], __shfl_xor_sync(0xffffffffu, cmax[j], 4));
      cmax[j] = fmaxf(cmax[j], __shfl_xor_sync(0xffffffffu, cmax[j], 8));
      cmax[j] = fmaxf(cmax[j], __shfl_xor_sync(0xffffffffu, cmax[j], 16));
    }
    float alpha[2], mnew[2], psum[2] = {0.f, 0.f}, pv[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      mnew[j] = fmaxf(mrun[j], cmax[j]);
      alpha[j] = ex2_approx(mrun[j] - mnew[j]);
    }
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = e & 1;
        pv[mt][e] = ex2_approx(x[mt][e] - mnew[j]);
        psum[j] += pv[mt][e];
      }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      lrun[j] = lrun[j] * alpha[j] + psum[j];
      mrun[j] = mnew[j];
    }

    // ---- P.V: k steps of 16 tokens (kk), A = V^T by movmatrix, B = P^T (P's
    // score fragments, split into fp16 pairs and transposed by movmatrix).
    // The chunk's products accumulate in fresh registers (4 MMAs deep), then
    // o = o * alpha + chunk in fp32 round to nearest.
    float cacc[2 * F::NB][4];
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      uint32_t bh0, bl0, bh1, bl1;
      {
        // lane (r, c) holds P of token 16kk + r (+ 8) for heads 2c, 2c+1: an
        // 8 x 8 (token, head) fragment; its transpose gives lane (r, c) head r
        // at tokens 2c, 2c+1 (+ 8), the B fragment
        uint32_t h0, l0, h1, l1;
        split_half2(pv[kk][0] * kPScale, pv[kk][1] * kPScale, h0, l0);
        split_half2(pv[kk][2] * kPScale, pv[kk][3] * kPScale, h1, l1);
        bh0 = movmatrix_t(h0);
        bl0 = movmatrix_t(l0);
        bh1 = movmatrix_t(h1);
        bl1 = movmatrix_t(l1);
      }
      const int ta = t0 + 16 * kk + r, tb = ta + 8;  // this lane's tokens in the movmatrix inputs
      const uint8_t* ra = vs_base + (16 * kk + r) * F::RB;
      const uint8_t* rb = ra + 8 * F::RB;
#pragma unroll
      for (int kb = 0; kb < F::NB; ++kb) {
        uint32_t va[4], vb[4];
        const int alc = row_align<V, D>(kb * F::BB), als = row_align<V, D>(kb * F::BB + 16);
        decode4(lds_bytes4_al(ra + kb * F::BB + 4 * c, alc), block_scales<V>(ra + kb * F::BB, als), va);
        decode4(lds_bytes4_al(rb + kb * F::BB + 4 * c, alc), block_scales<V>(rb + kb * F::BB, als), vb);
        if (t0 + kChunk > T) {  // only the last chunk has tokens past the sequence
#pragma unroll
          for (int k = 0; k < 4; ++k) {  // tokens past the sequence: zeros (their rows are not data)
            va[k] = ta < T ? va[k] : 0u;
            vb[k] = tb < T ? vb[k] : 0u;
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t a[4] = {movmatrix_t(va[2 * h]), movmatrix_t(va[2 * h + 1]), movmatrix_t(vb[2 * h]),
                                 movmatrix_t(vb[2 * h + 1])};
          if (kk == 0)  // the first step starts from zero
            mma_z(cacc[2 * kb + h], a, bh0, bh1, false);
          else
            mma_f16(cacc[2 * kb + h], a, bh0, bh1);
          mma_f16(cacc[2 * kb + h], a, bl0, bl1);
        }
      }
    }
#pragma unroll
    for (int m = 0; m < 2 * F::NB; ++m) {
      oacc[m][0] = fmaf(oacc[m][0], alpha[0], cacc[m][0]);
      oacc[m][1] = fmaf(oacc[m][1], alpha[1], cacc[m][1]);
      oacc[m][2] = fmaf(oacc[m][2], alpha[0], cacc[m][2]);
      oacc[m][3] = fmaf(oacc[m][3], alpha[1], cacc[m][3]);
    }
    __syncwarp();
    fence_proxy_async();  // the ring's reads precede the next bulk copy into it
    if (issued < n_mine) {
      issue(c0 + warp + issued * kAttnWarps, issued % kAttnStages);
      ++issued;
    }
  }
  if (!ok) {
    if (lane == 0) atomicOr(p.err, kErrWaitTimeout);
    for (int k = 0; k < issued; ++k) (void)mbar_wait_bounded(smem_addr(&bars[k % kAttnStages]), (uint32_t)((k / kAttnStages) & 1));
  }

  // the running sums of the 8 lanes of each head pair (fixed order)
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    lrun[j] += __shfl_xor_sync(0xffffffffu, lrun[j], 4);
    lrun[j] += __shfl_xor_sync(0xffffffffu, lrun[j], 8);
    lrun[j] += __shfl_xor_sync(0xffffffffu, lrun[j], 16);
  }

  // ---- merge the warps' states (warp order), then output or split partial ----
  __syncthreads();  // every ring is idle: the merge area reuses them
  float* mw = reinterpret_cast<float*>(smem) + (size_t)warp * partial_floats(D);
  if (r == 0) {
    mw[2 * c] = mrun[0];
    mw[2 * c + 1] = mrun[1];
    mw[8 + 2 * c] = lrun[0];
    mw[8 + 2 * c + 1] = lrun[1];
  }
  // o^T fragment m = (block kb, half h): row r holds D index
  // 32 kb + 4 (r / 2) + 2 h + 16 (r % 2), row r + 8 the next one.
#pragma unroll
  for (int m = 0; m < 2 * F::NB; ++m) {
    const int kb = m / 2, h = m % 2;
    const int dlo = 32 * kb + 4 * (r / 2) + 2 * h + 16 * (r % 2), dhi = dlo + 1;
    float* o = mw + 16;
    o[(2 * c) * D + dlo] = oacc[m][0] * kPUnscale;
    o[(2 * c + 1) * D + dlo] = oacc[m][1] * kPUnscale;
    o[(2 * c) * D + dhi] = oacc[m][2] * kPUnscale;
    o[(2 * c + 1) * D + dhi] = oacc[m][3] * kPUnscale;
  }
  __syncthreads();
  const float* base = reinterpret_cast<const float*>(smem);
  for (int i = threadIdx.x; i < G * D; i += kAttnWarps * 32) {
    const int g = i / D, d = i % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, base[w * partial_floats(D) + g]);
    float O = 0.f, L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) {
        const float* pw = base + w * partial_floats(D);
        const float e = exp2f(pw[g] - M);
        O += e * pw[16 + g * D + d];
        L += e * pw[8 + g];
      }
    }
    if (S == 1) {
      p.out[((size_t)b * p.H + (size_t)hk * G + g) * D + d] = L > 0.f ? O / L : 0.f;
    } else {
      float* part = p.ws + ((size_t)bhk * S + split) * partial_floats(D);
      if (d == 0) {
        part[g] = M;
        part[8 + g] = L;
      }
      part[16 + g * D + d] = O;
    }
  }
  grid_launch_dependents();
}

// Merges the S split partials of each (sequence, query head).  A CTA takes
// 32 of D for one (sequence, head); its nw warps (up to 8, about one per 4
// splits) each sum a contiguous share of the splits (in split order) and the
// sums are added in warp order.
// The split weights exp2(m_s - max) live in shared memory.  Fixed order
// throughout, so results are bitwise repeatable.
constexpr int kCombineWarps = 8;

RF4_DEV float block_max(float v, float* red, int nw) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float m = red[0];
  for (int i = 1; i < nw; ++i) m = fmaxf(m, red[i]);
  __syncthreads();
  return m;
}

template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32) attn_combine_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ float esh[];  // [S] split weights
  __shared__ float red[kCombineWarps][32];
  __shared__ float lsum;
  grid_dependency_wait();
  const int bh = blockIdx.x, d = blockIdx.y * 32 + (threadIdx.x & 31), w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int b = bh / p.H, h = bh % p.H, hk = h / p.G, g = h % p.G, S = p.S;
  const size_t PF = partial_floats(D);
  const float* base = p.ws + (size_t)(b * p.Hkv + hk) * S * PF;
  float m = -INFINITY;
  for (int s = threadIdx.x; s < S; s += nw * 32) m = fmaxf(m, base[s * PF + g]);
  const float M = block_max(m, &red[0][0], nw);
  for (int s = threadIdx.x; s < S; s += nw * 32) esh[s] = M == -INFINITY ? 0.f : exp2f(base[s * PF + g] - M);
  __syncthreads();
  if (w == 0) {
    // L = sum_s e_s l_s: lane l sums s = l, l + 32, ... in order, then a fixed shuffle tree
    float l = 0.f;
    for (int s = threadIdx.x; s < S; s += 32) l += esh[s] * base[s * PF + 8 + g];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (threadIdx.x == 0) lsum = l;
  }
  const int s0 = (int)((int64_t)w * S / nw), s1 = (int)((int64_t)(w + 1) * S / nw);
  float o = 0.f;
#pragma unroll 4
  for (int s = s0; s < s1; ++s) o += esh[s] * base[s * PF + 16 + g * D + d];
  red[w][threadIdx.x & 31] = o;
  __syncthreads();
  if (w == 0) {
    float O = red[0][threadIdx.x];
    for (int i = 1; i < nw; ++i) O += red[i][threadIdx.x];
    const float L = lsum;
    p.out[(size_t)bh * D + d] = L > 0.f ? O / L : 0.f;
  }
}

template <int V, int ACT>
const void* split_kernel_for(int D) {
  return D == 64 ? (const void*)&attn_split_kernel<V, ACT, 64> : (const void*)&attn_split_kernel<V, ACT, 128>;
}

const void* split_kernel(int variant, int act, int D) {
  if (variant == 0) return act == 0 ? split_kernel_for<0, 0>(D) : split_kernel_for<0, 1>(D);
  return act == 0 ? split_kernel_for<1, 0>(D) : split_kernel_for<1, 1>(D);
}

int split_smem(int variant, int D) {
  if (variant == 0) return D == 64 ? AttnFmt<0, 64>::SMEM : AttnFmt<0, 128>::SMEM;
  return D == 64 ? AttnFmt<1, 64>::SMEM : AttnFmt<1, 128>::SMEM;
}

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

// Split partials: groups * S < 2 * sms + groups < 4 * sms whenever the cache is split.
size_t attn_ws_floats(int sms) { return (size_t)4 * sms * partial_floats(kAttnMaxD); }

cudaError_t attn_prepare() {
  for (int v = 0; v < 2; ++v)
    for (int a = 0; a < 2; ++a)
      for (int D : {64, 128}) {
        cudaError_t e = cudaFuncSetAttribute(split_kernel(v, a, D), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             split_smem(v, D));
        if (e != cudaSuccess) return e;
      }
  return cudaSuccess;
}

cudaError_t launch_decode_attention(int variant, int act, const AttnArgs& a, int sms, cudaStream_t s, int* launches) {
  AttnParams p;
  p.q = a.q;
  p.K = a.K;
  p.V = a.V;
  p.lens = a.lens;
  p.out = a.out;
  p.ws = a.ws;
  p.B = (int)a.B;
  p.H = (int)a.H;
  p.Hkv = (int)a.Hkv;
  p.G = (int)(a.H / a.Hkv);
  p.Tmax = (int)a.Tmax;
  p.scale_log2 = a.scale * kLog2e;
  p.err = a.err;
  // Splits: about two CTAs per SM, at least 4 chunks of the cache per split
  // (measured against one and four per SM).
  const int64_t groups = a.B * a.Hkv;
  int64_t S = 1;
  if (groups < 2 * (int64_t)sms) {
    S = (2 * (int64_t)sms + groups - 1) / groups;
    const int64_t cap = a.Tmax / (4 * kChunk) > 1 ? a.Tmax / (4 * kChunk) : 1;
    S = S < cap ? S : cap;
  }
  p.S = (int)S;
  void* args[] = {&p};
  cudaError_t e = launch_pdl(split_kernel(variant, act, (int)a.D), dim3((unsigned)(groups * S)), dim3(kAttnWarps * 32),
                             split_smem(variant, (int)a.D), s, args);
  if (e != cudaSuccess) return e;
  *launches = 1;
  if (S == 1) return cudaSuccess;
  const void* comb = a.D == 64 ? (const void*)&attn_combine_kernel<64> : (const void*)&attn_combine_kernel<128>;
  const int nw = (int)((S + 3) / 4 < kCombineWarps ? (S + 3) / 4 : kCombineWarps);
  e = launch_pdl(comb, dim3((unsigned)(a.B * a.H), (unsigned)(a.D / 32)), dim3(nw * 32), sizeof(float) * (size_t)S, s,
                 args);
  if (e == cudaSuccess) *launches = 2;
  return e;
}

}  // namespace rocmfp4
