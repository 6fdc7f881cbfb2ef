// Streaming ROCmFP4 GEMV / small-batch product on sm_103a.
//
//   Y[m][n] = sum_k w[n][k] * X[m][k],  m < M <= 8,  fp32 accumulation.
//
// Decode path: "Feasibility Report: Porting ROCmFP4 to Atlas", section "What
// is ROCmFP4?" (Block Layout, Codebook10 Value Table, Scale Format); common.cuh
// explains how the Blackwell e2m1/e4m3 conversions reproduce it exactly.
//
// Work decomposition.  The matrix is cut into units of 32 rows x SPAN bytes
// (8 dual blocks = 144 B, or 16 single-scale blocks = 272 B, per row).
// Units are ordered tile-major (all K spans of rows 0..31, then rows 32..63,
// ...) and every active warp takes an equal contiguous range of them, four
// warps to a CTA.  The host sizes the grid (api.cu): one CTA per run of whole
// tiles when that keeps each CTA's weights small (then a tile is split only
// between the warps of one CTA), else every warp that fits.  A warp streams
// its units through a private ring of shared-memory stages: one 2-D TMA box
// of the unit's 32 weight rows plus a bulk copy per activation row of the
// unit's K span, one mbarrier per stage.  The DEEP instance has a deeper
// ring (two CTAs per SM) for grids that place at most two CTAs on an SM.
//
// Per unit, lane (q = lane/4, c = lane%4) owns rows q, q+8, q+16, q+24 (two
// m16 tiles that share every B fragment) and the 4-byte-aligned lane span c
// (BPL whole blocks) of each row.  Each block is eight mma.m16n8k16 steps:
// step s feeds qs bytes 2s and 2s+1 of the lane's block; each byte becomes
// one f16x2 A register (low nibble -> weight 2s or 2s+1 of half 0, high
// nibble -> the weight 16 further on, in half 1).  For M = 1 the 8 B columns
// hold (block, half) pairs, so each lane receives exact half-block sums and
// applies the fp32 half-scales once per half; for M > 1, B column n holds
// activation vector n (zero for n >= M) and the A registers carry the
// half-scales.  D is flushed into round-to-nearest fp32 registers after every
// block (8 MMAs), so the tensor core's own accumulation never runs long.
//
// A tile (32 rows) whose units are split between warps is finished by its
// last-arriving warp, in two levels: the warps of one CTA meet in shared
// memory, and CTAs that share a tile write 32 x 8 partials to the workspace,
// fence, and bump a per-tile counter; the one that completes the count sums
// all partials in K order, writes Y and resets the counter.  Nobody waits and
// the sum order is fixed, so results are bitwise reproducible.
#include <cudaTypedefs.h>

#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace rocmfp4 {
namespace {

constexpr int kWarps = kStreamWarpsPerCta;
constexpr int kTileRows = 32;  // rows per unit / tile: two m16 MMA tiles sharing each B fragment
constexpr int kRecFloats = kTileRows * 8;  // a global record: 32 rows x 8 columns

// Shared-memory part of the reduction (MB <= 4): kWarps x 2 records of
// 32 rows x MB columns, then one counter per warp.  A tile with parts in two
// or more warps of a CTA continues from its first such warp w into w + 1, and
// is w's last tile; so w identifies it.  With MB = 8 the records would cost
// the kernel a CTA per SM, and every warp uses the global level directly.
template <int MB>
constexpr size_t cta_red_bytes() {
  return MB <= 4 ? (size_t)kWarps * 2 * kTileRows * MB * 4 + kWarps * 4 : 0;
}


// Per-warp ring stage.  MB = 1: 32 weight rows x SPAN bytes, then the unit's
// KU activations.  MB >= 2 (M rounded up to 2, 4 or 8): first the unit's
// slice of MB activation rows, KU fp16/bf16 values each, as one tensor copy
// with the 128-byte swizzle (its 16-byte chunks XOR-permuted within each
// 1024 bytes, so that the lanes' fragment loads hit distinct banks: without
// it the eight rows of a load all fall in the same banks), then the weights;
// the stage is a multiple of 1024 bytes, as the swizzle needs.
template <int V, int MB>
constexpr int x_offset() { return MB == 1 ? kTileRows * Fmt<V>::SPAN : 0; }
template <int V, int MB>
constexpr int w_offset() { return MB == 1 ? 0 : MB * Fmt<V>::KU * 2; }
template <int V, int MB>
constexpr int stage_bytes() {
  return MB == 1 ? kTileRows * Fmt<V>::SPAN + Fmt<V>::KU * 2
                 : (MB * Fmt<V>::KU * 2 + kTileRows * Fmt<V>::SPAN + 1023) / 1024 * 1024;
}
// Slack for aligning the rings to 1024 bytes (MB >= 2).
template <int MB>
constexpr int ring_align_slack() { return MB == 1 ? 0 : 1024; }

// Chunk k (16 bytes) of block `blk` (64 bytes of activations) of row q in a
// swizzled activation slice: the logical offset's 16-byte chunk index XORed
// with its 128-byte line index modulo 8.
template <int V>
RF4_DEV const uint4* x_chunk(const uint8_t* xs, int q, int blk, int k) {
  const uint32_t off = (uint32_t)q * (Fmt<V>::KU * 2) + (uint32_t)blk * 64u + (uint32_t)k * 16u;
  return reinterpret_cast<const uint4*>(xs + (off ^ (((off >> 7) & 7u) << 4)));
}

// Stages per warp: as many as fit in about 54 KB per CTA (four CTAs, 16 warps
// per SM), at least 2 (one unit in flight while the previous one computes).
// DEEP = 1: about 108 KB per CTA (two CTAs per SM), for grids that place at
// most two CTAs on an SM: more of a small matrix is in flight, and more of it
// streams before the preceding grid ends.
template <int V, int MB, int DEEP = 0>
constexpr int stages() {
  constexpr int n = ((DEEP ? 108 : 54) * 1024) / (kWarps * stage_bytes<V, MB>());
  return n < 2 ? 2 : (n > 8 ? 8 : n);
}

constexpr int kZeroBytes = 256;  // zero activations for lanes whose B column is unused

template <int V, int MB, int DEEP = 0>
constexpr size_t smem_bytes() {
  return (size_t)ring_align_slack<MB>() + (size_t)kWarps * stages<V, MB, DEEP>() * stage_bytes<V, MB>() +
         (size_t)kWarps * stages<V, MB, DEEP>() * 8 + cta_red_bytes<MB>() + kZeroBytes;
}

__device__ __forceinline__ int64_t owner_of(int64_t u, int64_t U, int64_t wact) {
  return ((u + 1) * wact - 1) / U;
}

// E2M1 pair of the byte at (unrolled, hence constant) position pos of a word array.
template <int SW>
RF4_DEV uint32_t e2m1x2_at(const uint32_t (&w)[SW], int pos) {
  const uint32_t word = w[pos >> 2];
  switch (pos & 3) {
    case 0: return e2m1x2<0>(word);
    case 1: return e2m1x2<1>(word);
    case 2: return e2m1x2<2>(word);
    default: return e2m1x2<3>(word);
  }
}

// Scale pair of block phi of a lane span (f16x2 of the E4M3 values).
template <int V, int SW>
RF4_DEV uint32_t scale_pair_at(const uint32_t (&w)[SW], int phi) {
  const int P = phi * Fmt<V>::BB + 16;
  if constexpr (V == 0) {
    return (P & 2) ? e4m3x2<1>(w[P >> 2]) : e4m3x2<0>(w[P >> 2]);
  } else {
    const uint32_t dup = __byte_perm(w[P >> 2], 0u, (uint32_t)(P & 3) * 0x11u);
    return e4m3x2<0>(dup);
  }
}

// Codebook10 / 2 of a byte's two codes (no scale), in the MMA operand type.
template <int ACT>
RF4_DEV uint32_t code_pair(uint32_t codes_f16x2) {
  const uint32_t w = clamp5(codes_f16x2);
  if constexpr (ACT == 1) return f16x2_to_bf16x2(w);
  return w;
}

// E4M3 values of the scale pair of block phi of a lane span, as fp32.
template <int V, int SW>
RF4_DEV float2 scale_pair_f32(const uint32_t (&w)[SW], int phi) {
  const uint32_t h = scale_pair_at<V>(w, phi);
  const __half2 v = *reinterpret_cast<const __half2*>(&h);
  return make_float2(__low2float(v), __high2float(v));
}

template <int ACT>
RF4_DEV uint32_t weight_pair(uint32_t codes_f16x2, uint32_t s2) {
  const uint32_t w = hmul2(clamp5(codes_f16x2), s2);
  if constexpr (ACT == 1) return f16x2_to_bf16x2(w);
  return w;
}

// Copies of unit (t, j) into a stage: one 2-D tensor copy of the 32 x SPAN
// weight box (rows past N arrive as zeros) by lane 0, which also arms the
// stage's barrier for the whole unit; then lanes 0..M-1 copy the unit's slice
// of one activation row each (issue_x).
template <int V, int MB, int EPI>
__device__ __forceinline__ void issue_w(const CUtensorMap* tmw, int M, int t, int j, uint8_t* stage, uint32_t bar,
                                        int lane) {
  using F = Fmt<V>;
  if (lane == 0) {
    // MB >= 2: the activation box has MB rows (rows past M arrive as zeros)
    mbar_arrive_expect_tx(bar, (uint32_t)(kTileRows * F::SPAN + (MB == 1 ? M : MB) * F::KU * 2));
    uint8_t* dst = stage + w_offset<V, MB>();
    if constexpr (EPI)  // box {span, 16 rows, gate and up halves}: gate rows land in rows 0-15, up rows in 16-31
      tma_load_3d(smem_addr(dst), tmw, j * (F::SPAN / 4), t * (kTileRows / 2), 0, bar);
    else
      tma_load_2d(smem_addr(dst), tmw, j * (F::SPAN / 4), t * kTileRows, bar);
  }
}

template <int V, int MB>
__device__ __forceinline__ void issue_x(const uint16_t* __restrict__ X, const CUtensorMap* tmx, int j, uint8_t* stage,
                                        uint32_t bar, int lane) {
  using F = Fmt<V>;
  if (lane != 0) return;
  if constexpr (MB == 1)
    bulk_g2s(smem_addr(stage + x_offset<V, MB>()), X + (int64_t)j * F::KU, F::KU * 2, bar);
  else  // box {64 values, KU / 64 lines, MB rows} at line j * KU / 64, swizzled
    tma_load_3d(smem_addr(stage + x_offset<V, MB>()), tmx, 0, j * (F::KU / 64), 0, bar);
}

// One product of a launch.  The tensor map views the weights as N rows of
// row_bytes / 4 32-bit words, with a box of SPAN / 4 words x 32 rows.
struct StreamOp {
  CUtensorMap tmw;
  CUtensorMap tmx;  // activations as {64 values, K / 64 lines, M rows}, 128-byte swizzle (M >= 2)
  const uint16_t* X;
  float* Y;
  int64_t N, K, units, nspans;
  int64_t wact;  // warps sharing this product's units (<= units and <= the launch's warps)
};

// Parameters of a launch.
struct StreamParams {
  StreamOp op;
  float* ws;       // 2 * wact records of 32 x 8 floats
  uint32_t* cnt;   // split-tile counters, zero between launches
  uint32_t* err;   // error bits
  int M;
};

// Adds one unit's products into acc (see the kernel comment for the layouts).
// Lanes whose B column carries no activations read theirs from `zero`, a
// 256-byte page of zeros in shared memory, so every lane runs the same loads.
template <int V, int ACT, int MB>
RF4_DEV void compute_unit(const uint8_t* stage, int lane, int M, float (&acc)[2][4], const uint4* zero) {
  using F = Fmt<V>;
  constexpr int SW = F::SW;
  const int q = lane >> 2, c = lane & 3;
  const uint8_t* sb = stage + w_offset<V, MB>() + c * F::LANE_BYTES;
  // rows q, q+8 (m-tile 0) and q+16, q+24 (m-tile 1): words of the lane span,
  // loaded inside each block's step (only that block's words stay live)
  auto load_words = [&](uint32_t (&w0)[SW], uint32_t (&w1)[SW], uint32_t (&w2)[SW], uint32_t (&w3)[SW]) {
#pragma unroll
    for (int k = 0; k < SW; ++k) {
      w0[k] = reinterpret_cast<const uint32_t*>(sb + q * F::SPAN)[k];
      w1[k] = reinterpret_cast<const uint32_t*>(sb + (q + 8) * F::SPAN)[k];
      w2[k] = reinterpret_cast<const uint32_t*>(sb + (q + 16) * F::SPAN)[k];
      w3[k] = reinterpret_cast<const uint32_t*>(sb + (q + 24) * F::SPAN)[k];
    }
  };
  if constexpr (MB == 1) {
    // M == 1, column split: B column n = 2c' + h holds x only for the k rows
    // of lane c''s block and half h, so D[row][2c + h] is the half-block sum
    // sum_i (Codebook10[q_i] / 2) * x_i of lane c's block.  Lane (q, c) thus
    // holds exactly its own block's half sums for rows q, q+8 (per m-tile),
    // and applies the scales once per half-block in fp32.
    const int hb = q & 1;
    const bool bact = (q >> 1) == c;
    const uint32_t sel0 = !bact ? 0x4444u : (hb ? 0x1044u : 0x4410u);  // (x[2s], 0) or (0, x[2s+16])
    const uint32_t sel1 = !bact ? 0x4444u : (hb ? 0x3244u : 0x4432u);  // (x[2s+1], 0) or (0, x[2s+17])
    // the 16 activations of half hb of block c*BPL + phi at xp[phi * 4 + 0..1]
    const uint4* xp = bact ? reinterpret_cast<const uint4*>(stage + x_offset<V, MB>()) + c * F::BPL * 4 + 2 * hb
                           : zero;
#pragma unroll
    for (int phi = 0; phi < F::BPL; ++phi) {
      uint32_t w0[SW], w1[SW], w2[SW], w3[SW];
      load_words(w0, w1, w2, w3);
      uint32_t xh[8];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const uint4 v = xp[phi * 4 + k];
        xh[4 * k] = v.x;
        xh[4 * k + 1] = v.y;
        xh[4 * k + 2] = v.z;
        xh[4 * k + 3] = v.w;
      }
      float d0[4], d1[4];
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int pos = phi * F::BB + 2 * s;
        const uint32_t b0 = __byte_perm(xh[s], 0u, sel0);
        const uint32_t b1 = __byte_perm(xh[s], 0u, sel1);
        uint32_t a[4];
        a[0] = code_pair<ACT>(e2m1x2_at(w0, pos));
        a[1] = code_pair<ACT>(e2m1x2_at(w1, pos));
        a[2] = code_pair<ACT>(e2m1x2_at(w0, pos + 1));
        a[3] = code_pair<ACT>(e2m1x2_at(w1, pos + 1));
        if (s == 0) mma16816_z(d0, a, b0, b1, ACT == 1);
        else mma16816(d0, a, b0, b1, ACT == 1);
        a[0] = code_pair<ACT>(e2m1x2_at(w2, pos));
        a[1] = code_pair<ACT>(e2m1x2_at(w3, pos));
        a[2] = code_pair<ACT>(e2m1x2_at(w2, pos + 1));
        a[3] = code_pair<ACT>(e2m1x2_at(w3, pos + 1));
        if (s == 0) mma16816_z(d1, a, b0, b1, ACT == 1);
        else mma16816(d1, a, b0, b1, ACT == 1);
      }
      // E4M3 values of the scales of the lane's block, rows q, q+8, q+16, q+24
      const float2 e0 = scale_pair_f32<V>(w0, phi), e1 = scale_pair_f32<V>(w1, phi);
      const float2 e2 = scale_pair_f32<V>(w2, phi), e3 = scale_pair_f32<V>(w3, phi);
      acc[0][0] = fmaf(d0[0], e0.x, acc[0][0]);
      acc[0][1] = fmaf(d0[1], e0.y, acc[0][1]);
      acc[0][2] = fmaf(d0[2], e1.x, acc[0][2]);
      acc[0][3] = fmaf(d0[3], e1.y, acc[0][3]);
      acc[1][0] = fmaf(d1[0], e2.x, acc[1][0]);
      acc[1][1] = fmaf(d1[1], e2.y, acc[1][1]);
      acc[1][2] = fmaf(d1[2], e3.x, acc[1][2]);
      acc[1][3] = fmaf(d1[3], e3.y, acc[1][3]);
    }
  } else {
    // D accumulates the whole unit (2 dual or 4 single-scale blocks = 16 or
    // 32 MMAs) and is then flushed into round-to-nearest fp32 registers.
    // Lane (q, c) holds B column q: activation row q, or zeros for q >= M.
    const uint8_t* xs = stage + x_offset<V, MB>();
    const bool xrow = q < M;
    float d0[4], d1[4];
#pragma unroll
    for (int phi = 0; phi < F::BPL; ++phi) {
      // 32 activations of the lane's block (block c*BPL + phi of the unit)
      uint32_t w0[SW], w1[SW], w2[SW], w3[SW];
      load_words(w0, w1, w2, w3);
      uint32_t xv[16];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 v = xrow ? *x_chunk<V>(xs, q, c * F::BPL + phi, k) : zero[phi * 4 + k];
        xv[4 * k] = v.x;
        xv[4 * k + 1] = v.y;
        xv[4 * k + 2] = v.z;
        xv[4 * k + 3] = v.w;
      }
      const uint32_t s0 = scale_pair_at<V>(w0, phi), s1 = scale_pair_at<V>(w1, phi);
      const uint32_t s2 = scale_pair_at<V>(w2, phi), s3 = scale_pair_at<V>(w3, phi);
#pragma unroll
      for (int s = 0; s < 8; ++s) {
        const int pos = phi * F::BB + 2 * s;
        // B rows (2c, 2c+1) = (x[2s], x[2s+16]); rows (2c+8, 2c+9) = (x[2s+1], x[2s+17]).
        const uint32_t b0 = __byte_perm(xv[s], xv[8 + s], 0x5410);
        const uint32_t b1 = __byte_perm(xv[s], xv[8 + s], 0x7632);
        uint32_t a[4];
        a[0] = weight_pair<ACT>(e2m1x2_at(w0, pos), s0);
        a[1] = weight_pair<ACT>(e2m1x2_at(w1, pos), s1);
        a[2] = weight_pair<ACT>(e2m1x2_at(w0, pos + 1), s0);
        a[3] = weight_pair<ACT>(e2m1x2_at(w1, pos + 1), s1);
        if (phi == 0 && s == 0) mma16816_z(d0, a, b0, b1, ACT == 1);
        else mma16816(d0, a, b0, b1, ACT == 1);
        a[0] = weight_pair<ACT>(e2m1x2_at(w2, pos), s2);
        a[1] = weight_pair<ACT>(e2m1x2_at(w3, pos), s3);
        a[2] = weight_pair<ACT>(e2m1x2_at(w2, pos + 1), s2);
        a[3] = weight_pair<ACT>(e2m1x2_at(w3, pos + 1), s3);
        if (phi == 0 && s == 0) mma16816_z(d1, a, b0, b1, ACT == 1);
        else mma16816(d1, a, b0, b1, ACT == 1);
      }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      acc[0][r] += d0[r];
      acc[1][r] += d1[r];
    }
  }
}

// Split-tile reduction.  A tile (32 rows x all K) whose spans are spread over
// several warps is summed in two levels, each in a fixed order, so results
// are bitwise reproducible:
//   1. the warps of one CTA that hold parts of the tile add them in shared
//      memory: each writes a record (32 rows x 8 columns) and bumps a
//      per-tile shared counter; the last of them sums the records in warp
//      (= K) order;
//   2. if the tile also has parts in other CTAs, that warp writes the CTA's
//      sum as a record in global memory and bumps a per-tile global counter;
//      the last CTA sums the CTA records in CTA (= K) order and stores Y.
// Nobody waits: whoever completes a count does the sum.

struct CtaRed {
  float* rec;     // [kWarps][2][32 * MB]
  uint32_t* cnt;  // [kWarps], zero between tiles
};

// Record layout: row r, column m at rec[r * RS + m] (RS columns, M <= RS).
// From the MMA fragments of acc (owner lanes only write).
template <bool COL, int RS>
RF4_DEV void write_record_frag(float* rec, const float (&acc)[2][4], int lane) {
  const int q = lane >> 2, c = lane & 3;
  const int c0 = COL ? 0 : 2 * c, c1 = COL ? 1 : 2 * c + 1;
  if ((COL && c != 0) || c0 >= RS) return;
#pragma unroll
  for (int mt = 0; mt < 2; ++mt) {
    const int r0 = mt * 16 + q;
    rec[r0 * RS + c0] = acc[mt][0];
    rec[(r0 + 8) * RS + c0] = acc[mt][2];
    if (!COL) {
      rec[r0 * RS + c1] = acc[mt][1];
      rec[(r0 + 8) * RS + c1] = acc[mt][3];
    }
  }
}

// Record layout from row-per-lane sums (lane r holds row r).
template <int RS>
RF4_DEV void write_record_rows(float* rec, const float (&sum)[8], int lane, int M) {
  if (M == 1) {
    rec[lane * RS] = sum[0];
  } else if constexpr (RS % 4 == 0) {
#pragma unroll
    for (int h = 0; h < RS / 4; ++h)
      reinterpret_cast<float4*>(rec + lane * RS)[h] =
          make_float4(sum[4 * h], sum[4 * h + 1], sum[4 * h + 2], sum[4 * h + 3]);
  } else {
#pragma unroll
    for (int m = 0; m < RS; ++m) rec[lane * RS + m] = sum[m];
  }
}

// Row-per-lane sum of records first .. last (in that order) at
// base + (2 * (idx - idx0) + slot) * 32 * RS; record `first` is in slot
// `slot_first`, the others in slot 0.  Global records are read through L2.
template <bool GLOBAL, int RS>
RF4_DEV void sum_records(const float* base, int64_t idx0, int64_t first, int64_t last, int slot_first, int lane, int M,
                         float (&sum)[8]) {
  constexpr int RF = kTileRows * RS;
#pragma unroll
  for (int m = 0; m < 8; ++m) sum[m] = 0.f;
  if (M == 1) {
    for (int64_t w0 = first; w0 <= last; w0 += 8) {
      float v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int64_t w = w0 + k;
        const float* r = base + (2 * (w - idx0) + (w == first ? slot_first : 0)) * RF + lane * RS;
        v[k] = w <= last ? (GLOBAL ? __ldcg(r) : *r) : 0.f;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (w0 + k <= last) sum[0] += v[k];
    }
  } else {
    // RS = 2, 4 or 8 columns per row: 8-, 16- or 32-byte aligned, read as vectors
    for (int64_t w0 = first; w0 <= last; w0 += 4) {
      float v[4][RS];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int64_t w = w0 + k;
        const float* r = base + (2 * (w - idx0) + (w == first ? slot_first : 0)) * RF + lane * RS;
        if (w <= last) {
          if constexpr (RS == 2) {
            const float2 a = GLOBAL ? __ldcg(reinterpret_cast<const float2*>(r)) : *reinterpret_cast<const float2*>(r);
            v[k][0] = a.x;
            v[k][1] = a.y;
          } else {
#pragma unroll
            for (int h = 0; h < RS / 4; ++h) {
              const float4* r4 = reinterpret_cast<const float4*>(r) + h;
              const float4 a = GLOBAL ? __ldcg(r4) : *r4;
              v[k][4 * h] = a.x;
              v[k][4 * h + 1] = a.y;
              v[k][4 * h + 2] = a.z;
              v[k][4 * h + 3] = a.w;
            }
          }
        } else {
#pragma unroll
          for (int m = 0; m < RS; ++m) v[k][m] = 0.f;
        }
      }
#pragma unroll
      for (int k = 0; k < 4; ++k)
        if (w0 + k <= last)
#pragma unroll
          for (int m = 0; m < RS; ++m) sum[m] += v[k][m];
    }
  }
}

// SiLU(g) = g / (1 + exp(-g)) with the fast exponential and division (no
// slow-path subroutine in the kernel): relative error a few 1e-6 where the
// gate is not saturated; very negative g (exp(-g) = inf) gives 0.
RF4_DEV float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Stores tile t from row-per-lane sums (lane r holds row r of the tile).  In
// gate/up mode lanes 0-15 hold the gate rows and 16-31 the up rows of the
// tile's 16 outputs.  Every lane of the warp must call it.
template <int EPI>
RF4_DEV void store_rows(float* __restrict__ Y, int64_t N, int64_t t, int lane, const float (&sum)[8], int M) {
  if constexpr (EPI) {
    float up[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) up[m] = __shfl_down_sync(0xffffffffu, sum[m], 16);
    const int64_t o = t * (kTileRows / 2) + lane;
    if (lane < 16 && o < N)
#pragma unroll
      for (int m = 0; m < 8; ++m)
        if (m < M) Y[m * N + o] = silu(sum[m]) * up[m];
    return;
  }
  const int64_t row = t * kTileRows + lane;
  if (row < N)
#pragma unroll
    for (int m = 0; m < 8; ++m)
      if (m < M) Y[m * N + row] = sum[m];
}

RF4_DEV uint32_t shared_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_addr(p)), "r"(v) : "memory");
  return old;
}

// End of tile t of product op for this warp (its spans [js, j] are in acc):
// store the tile if the warp covered all of it, else hand its partial to the
// split-tile reduction.  Resets acc.
template <int MB, int EPI>
RF4_DEV void finish_tile(const StreamParams& p, const StreamOp& op, int64_t wg, int t, int js, int j, int lane,
                         float (&acc)[2][4], const CtaRed& red) {
  constexpr bool COL = MB == 1;
  constexpr bool LOCAL = cta_red_bytes<MB>() > 0;  // level 1 in shared memory
  const int M = p.M;
  const int64_t N = op.N, S = op.nspans, U = op.units, wact = op.wact;
  float* __restrict__ Y = op.Y;
  const int q = lane >> 2, c = lane & 3;
  // Bring the partial sums to lanes: in column-split mode add the two halves
  // and the four lanes of each quad (fixed order), so lane (q, 0) holds rows
  // q, q+8, q+16, q+24.
  if constexpr (COL) {
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      float ra = acc[mt][0] + acc[mt][1], rb = acc[mt][2] + acc[mt][3];
      ra += __shfl_xor_sync(0xffffffffu, ra, 1);
      rb += __shfl_xor_sync(0xffffffffu, rb, 1);
      ra += __shfl_xor_sync(0xffffffffu, ra, 2);
      rb += __shfl_xor_sync(0xffffffffu, rb, 2);
      acc[mt][0] = ra;  // (Codebook10 / 2) x E4M3 = Codebook10 x half-scale
      acc[mt][2] = rb;
      acc[mt][1] = acc[mt][3] = 0.f;
    }
  }
  if (js == 0 && j == S - 1) {
    // the whole tile is this warp's
    const int c0 = COL ? 0 : 2 * c, c1 = COL ? 1 : 2 * c + 1;
    if constexpr (EPI) {
      // m-tile 0 holds the gate rows, m-tile 1 the up rows of the same outputs
      if (!COL || c == 0) {
        const int64_t oa = (int64_t)t * (kTileRows / 2) + q, ob = oa + 8;
        if (c0 < M) {
          if (oa < N) Y[c0 * N + oa] = silu(acc[0][0]) * acc[1][0];
          if (ob < N) Y[c0 * N + ob] = silu(acc[0][2]) * acc[1][2];
        }
        if (!COL && c1 < M) {
          if (oa < N) Y[c1 * N + oa] = silu(acc[0][1]) * acc[1][1];
          if (ob < N) Y[c1 * N + ob] = silu(acc[0][3]) * acc[1][3];
        }
      }
    } else if (!COL || c == 0) {
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const int64_t ra = (int64_t)t * kTileRows + mt * 16 + q, rb = ra + 8;
        if (c0 < M) {
          if (ra < N) Y[c0 * N + ra] = acc[mt][0];
          if (rb < N) Y[c0 * N + rb] = acc[mt][2];
        }
        if (!COL && c1 < M) {
          if (ra < N) Y[c1 * N + ra] = acc[mt][1];
          if (rb < N) Y[c1 * N + rb] = acc[mt][3];
        }
      }
    }
  } else {
    const int64_t tS = (int64_t)t * S;
    const int64_t wf = owner_of(tS, U, wact), wl = owner_of(tS + S - 1, U, wact);  // the tile's warps
    const int64_t cta = wg / kWarps, w0c = cta * kWarps;
    const int64_t wlast_cta = (w0c + kWarps < wact ? w0c + kWarps : wact) - 1;
    const int64_t lf = wf > w0c ? wf : w0c, ll = wl < wlast_cta ? wl : wlast_cta;  // the tile's warps in this CTA
    const int slot_wf = U * wf / wact < tS ? 1 : 0;  // the first warp started before the tile
    const int key = (int)(lf - w0c);
    float sum[8];
    bool pass = true;     // this warp carries the CTA's part on
    bool rows = false;    // ... as row-per-lane sums (else as fragments in acc)
    if (LOCAL && ll > lf) {
      // level 1: the CTA's warps meet in shared memory
      write_record_frag<COL, MB>(red.rec + ((wg - w0c) * 2 + (wg == wf ? slot_wf : 0)) * (kTileRows * MB), acc, lane);
      __syncwarp();
      uint32_t old = 0;
      if (lane == 0) old = shared_add_acq_rel(&red.cnt[key], 1u);
      old = __shfl_sync(0xffffffffu, old, 0);
      pass = (int64_t)old == ll - lf;
      if (pass) {
        sum_records<false, MB>(red.rec, w0c, lf, ll, lf == wf ? slot_wf : 0, lane, M, sum);
        rows = true;
        __syncwarp();
        if (lane == 0) red.cnt[key] = 0u;
      }
    }
    if (pass) {
      // level 2 counts CTAs (or warps, without level 1)
      const int64_t per = LOCAL ? kWarps : 1;
      const int64_t me = wg / per, uf = wf / per, ul = wl / per;
      if (uf == ul) {
        // every part was in this CTA
        store_rows<EPI>(Y, N, t, lane, sum, M);
      } else {
        // one record per contributor in global memory, counted per tile
        const int slot_uf = U * (uf * per) / wact < tS ? 1 : 0;
        float* grec = p.ws + (2 * me + (me == uf ? slot_uf : 0)) * kRecFloats;
        if (rows) write_record_rows<8>(grec, sum, lane, M);
        else write_record_frag<COL, 8>(grec, acc, lane);
        __syncwarp();  // orders the warp's record stores before lane 0's release
        uint32_t old = 0;
        if (lane == 0) old = atomic_add_acq_rel_gpu(&p.cnt[uf], 1u);
        old = __shfl_sync(0xffffffffu, old, 0);  // lane 0's acquire is shared with the warp
        if ((int64_t)old == ul - uf) {
          sum_records<true, 8>(p.ws, 0, uf, ul, slot_uf, lane, M, sum);
          store_rows<EPI>(Y, N, t, lane, sum, M);
          __syncwarp();
          if (lane == 0) store_relaxed_gpu(&p.cnt[uf], 0u);
        }
      }
    }
  }
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int r = 0; r < 4; ++r) acc[mt][r] = 0.f;
}

// The streaming kernel of one product.  Each warp owns an equal contiguous
// range of the product's units (tile-major) and streams them through its
// ring.  Weights never depend on earlier work: up to NS - 1 units of them are
// requested before the programmatic-dependent-launch wait, so they stream
// while the preceding grid drains; activations, outputs and the split-tile
// workspace are touched only after the wait.
// EPI = 1: the gate/up mode.
template <int V, int ACT, int MB, int EPI, int DEEP>
__global__ void __launch_bounds__(kWarps * 32, 4) gemv_stream_kernel(const __grid_constant__ StreamParams p) {
  using F = Fmt<V>;
  constexpr int NS = stages<V, MB, DEEP>();
  constexpr int SB = stage_bytes<V, MB>();
  extern __shared__ __align__(128) uint8_t smem[];

  const StreamOp& op = p.op;
  const int M = p.M;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t wg = (int64_t)blockIdx.x * kWarps + warp;

  // the rings start on a 1024-byte boundary when the activations are swizzled
  uint8_t* const base = smem + (ring_align_slack<MB>() ? (1024u - (smem_addr(smem) & 1023u)) & 1023u : 0u);
  uint8_t* ring = base + (size_t)warp * NS * SB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + (size_t)kWarps * NS * SB) + warp * NS;
  // after every warp's stage barriers: the shared part of the split-tile
  // reduction, then a page of zeros
  CtaRed red;
  red.rec = reinterpret_cast<float*>(base + (size_t)kWarps * NS * SB + (size_t)kWarps * NS * 8);
  red.cnt = reinterpret_cast<uint32_t*>(red.rec + kWarps * 2 * kTileRows * MB);  // used only if cta_red_bytes<MB>() > 0
  uint4* zero = reinterpret_cast<uint4*>(base + (size_t)kWarps * NS * SB + (size_t)kWarps * NS * 8 + cta_red_bytes<MB>());
  if (threadIdx.x < kZeroBytes / 16) zero[threadIdx.x] = make_uint4(0u, 0u, 0u, 0u);
  if (cta_red_bytes<MB>() > 0 && threadIdx.x < kWarps) red.cnt[threadIdx.x] = 0u;
  __syncthreads();  // every thread of the CTA gets here: inactive warps return below
  if (wg >= op.wact) return;
  if (lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&op.tmw)) : "memory");
    for (int i = 0; i < NS; ++i) mbar_init(smem_addr(&bars[i]), 1);
    fence_mbar_init();
  }
  __syncwarp();

  // A single product: this warp's units u0 .. u1 - 1, tile-major.  Weights
  // of up to NS - 1 units are requested before the dependency wait; after
  // it, each unit's activations go out with (or right after) its weights.
  const int S = (int)op.nspans;
  const int64_t u0 = op.units * wg / op.wact, u1 = op.units * (wg + 1) / op.wact;
  const int n = (int)(u1 - u0);
  int tw = (int)(u0 / S), jw = (int)(u0 % S), jx = jw;
  int iw = 0, ix = 0, sw = 0, sx = 0;  // units issued (weights, activations) and their stages
  auto issue_w1 = [&]() {
    issue_w<V, MB, EPI>(&op.tmw, M, tw, jw, ring + (size_t)sw * SB, smem_addr(&bars[sw]), lane);
    if (++jw == S) {
      jw = 0;
      ++tw;
    }
    if (++sw == NS) sw = 0;
    ++iw;
  };
  auto issue_x1 = [&]() {
    issue_x<V, MB>(op.X, &op.tmx, jx, ring + (size_t)sx * SB, smem_addr(&bars[sx]), lane);
    if (++jx == S) jx = 0;
    if (++sx == NS) sx = 0;
    ++ix;
  };
  while (iw < NS - 1 && iw < n) issue_w1();
  grid_dependency_wait();
  grid_launch_dependents();
  __syncwarp();
  while (ix < iw) issue_x1();

  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  int t = (int)(u0 / S), j = (int)(u0 % S), js = j;
  int k = 0, st = 0;
  uint32_t phase = 0;
  bool failed = false;
  for (; k < n; ++k) {
    if (iw < n) {  // unit k + NS - 1 goes into the stage unit k - 1 has released
      issue_w1();
      issue_x1();
    }
    if (!mbar_wait_bounded(smem_addr(&bars[st]), phase)) {
      failed = true;
      break;
    }
    compute_unit<V, ACT, MB>(ring + (size_t)st * SB, lane, M, acc, zero);
    __syncwarp();
    fence_proxy_async();
    if (j == S - 1 || k == n - 1) {
      finish_tile<MB, EPI>(p, op, wg, t, js, j, lane, acc, red);
      js = 0;
    }
    if (++j == S) {
      j = 0;
      ++t;
    }
    if (++st == NS) {
      st = 0;
      phase ^= 1u;
    }
  }
  if (failed) {
    if (lane == 0) atomicOr(p.err, kErrWaitTimeout);
    // every armed stage has its activation copies issued (ix == iw); let all copies land
    for (; k < iw; ++k) {
      (void)mbar_wait_bounded(smem_addr(&bars[st]), phase);
      if (++st == NS) {
        st = 0;
        phase ^= 1u;
      }
    }
  }
}

// Kernel instance for (variant, activation type, staged activation rows,
// plain or gate/up).
template <int V, int ACT, int EPI>
const void* kernel_for_mb(int mb) {
  switch (mb) {
    case 1: return reinterpret_cast<const void*>(&gemv_stream_kernel<V, ACT, 1, EPI, 0>);
    case 2: return reinterpret_cast<const void*>(&gemv_stream_kernel<V, ACT, 2, EPI, 0>);
    case 4: return reinterpret_cast<const void*>(&gemv_stream_kernel<V, ACT, 4, EPI, 0>);
    default: return reinterpret_cast<const void*>(&gemv_stream_kernel<V, ACT, 8, EPI, 0>);
  }
}

// The deep-ring instance of a plain product (MB = 1 or 2 only).
template <int V, int ACT>
const void* deep_kernel_for_mb(int mb) {
  return mb == 1 ? reinterpret_cast<const void*>(&gemv_stream_kernel<V, ACT, 1, 0, 1>)
                 : reinterpret_cast<const void*>(&gemv_stream_kernel<V, ACT, 2, 0, 1>);
}

template <int EPI>
const void* plain_kernel(int variant, int act, int mb) {
  if (variant == 0) return act == 0 ? kernel_for_mb<0, 0, EPI>(mb) : kernel_for_mb<0, 1, EPI>(mb);
  return act == 0 ? kernel_for_mb<1, 0, EPI>(mb) : kernel_for_mb<1, 1, EPI>(mb);
}

// kind 0: plain product, 1: gate/up product, 2: plain product with the deep
// ring (MB <= 2).
const void* stream_kernel(int variant, int act, int mb, int kind) {
  if (kind == 2) {
    if (variant == 0) return act == 0 ? deep_kernel_for_mb<0, 0>(mb) : deep_kernel_for_mb<0, 1>(mb);
    return act == 0 ? deep_kernel_for_mb<1, 0>(mb) : deep_kernel_for_mb<1, 1>(mb);
  }
  return kind == 1 ? plain_kernel<1>(variant, act, mb) : plain_kernel<0>(variant, act, mb);
}

template <int V>
size_t smem_for_mb(int mb, int deep) {
  switch (mb) {
    case 1: return deep ? smem_bytes<V, 1, 1>() : smem_bytes<V, 1>();
    case 2: return deep ? smem_bytes<V, 2, 1>() : smem_bytes<V, 2>();
    case 4: return smem_bytes<V, 4>();
    default: return smem_bytes<V, 8>();
  }
}

}  // namespace

int stream_mb_for(int M) { return M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8; }

int stream_weights_per_unit(int variant) { return variant == 0 ? Fmt<0>::KU : Fmt<1>::KU; }

size_t stream_smem_bytes(int variant, int mb, int deep) {
  return variant == 0 ? smem_for_mb<0>(mb, deep) : smem_for_mb<1>(mb, deep);
}

cudaError_t stream_prepare(int variant, int act, int mb) {
  for (int kind = 0; kind < 3; ++kind) {
    if (kind == 2 && mb > 2) break;
    cudaError_t e =
        cudaFuncSetAttribute(stream_kernel(variant, act, mb, kind), cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)stream_smem_bytes(variant, mb, kind == 2 ? 1 : 0));
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t stream_occupancy(int variant, int act, int mb, int* ctas_per_sm) {
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, stream_kernel(variant, act, mb, 0),
                                                                kWarps * 32, stream_smem_bytes(variant, mb, 0));
  return e;
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
}

cudaError_t stream_init_driver() {
  if (g_encode) return cudaSuccess;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
  if (e != cudaSuccess) return e;
  if (q != cudaDriverEntryPointSuccess || fn == nullptr) return cudaErrorSymbolNotFound;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return cudaSuccess;
}

namespace {

cudaError_t encode_weights(int variant, const GemvArgs& a, CUtensorMap* tmw) {
  const int span = variant == 0 ? Fmt<0>::SPAN : Fmt<1>::SPAN;
  if (a.epi) {
    // Gate/up pairing: words x N rows x {gate, up}; a box takes 16 rows of each.
    cuuint64_t dims[3] = {(cuuint64_t)(a.row_bytes / 4), (cuuint64_t)a.N, 2};
    cuuint64_t strides[2] = {(cuuint64_t)a.row_bytes, (cuuint64_t)(a.row_bytes * a.N)};
    cuuint32_t box[3] = {(cuuint32_t)(span / 4), (cuuint32_t)(kTileRows / 2), 2};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(tmw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<uint8_t*>(a.W), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
  }
  // Weights as a 2-D array of 32-bit words: row_bytes/4 columns, N rows.
  cuuint64_t dims[2] = {(cuuint64_t)(a.row_bytes / 4), (cuuint64_t)a.N};
  cuuint64_t strides[1] = {(cuuint64_t)a.row_bytes};
  cuuint32_t box[2] = {(cuuint32_t)(span / 4), (cuuint32_t)kTileRows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(tmw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint8_t*>(a.W), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Activations of M >= 2 rows as {64 values, K / 64 lines of 128 bytes, M
// rows}; a box is one unit's slice of MB rows, with the 128-byte swizzle.
cudaError_t encode_acts(int variant, const GemvArgs& a, int mb, CUtensorMap* tmx) {
  const int ku = variant == 0 ? Fmt<0>::KU : Fmt<1>::KU;
  cuuint64_t dims[3] = {64, (cuuint64_t)(a.K / 64), (cuuint64_t)a.M};
  cuuint64_t strides[2] = {128, (cuuint64_t)a.K * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)(ku / 64), (cuuint32_t)mb};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(tmx, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint16_t*>(a.X), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t fill_params(int variant, const GemvArgs& a, StreamParams* p) {
  memset(p, 0, sizeof(*p));
  cudaError_t e = encode_weights(variant, a, &p->op.tmw);
  if (e != cudaSuccess) return e;
  const int mb = stream_mb_for(a.M);
  if (mb >= 2 && (e = encode_acts(variant, a, mb, &p->op.tmx)) != cudaSuccess) return e;
  p->op.X = a.X;
  p->op.Y = a.Y;
  p->op.N = a.N;
  p->op.K = a.K;
  p->op.units = a.units;
  p->op.nspans = a.nspans;
  p->op.wact = a.units < a.wact ? a.units : a.wact;
  p->ws = a.ws;
  p->cnt = a.cnt;
  p->err = a.err;
  p->M = a.M;
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemv_stream(int variant, int act, const GemvArgs& a, int ctas, cudaStream_t s) {
  if (!g_encode) return cudaErrorInitializationError;
  const int mb = stream_mb_for(a.M);
  StreamParams p;
  cudaError_t e = fill_params(variant, a, &p);
  if (e != cudaSuccess) return e;
  // Programmatic dependent launch: the kernel may start (and stream weights)
  // while the previous kernel on the stream drains; it calls
  // griddepcontrol.wait before reading anything an earlier kernel writes.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kWarps * 32);
  const int deep = a.deep && !a.epi && mb <= 2 ? 1 : 0;
  cfg.dynamicSmemBytes = stream_smem_bytes(variant, mb, deep);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&p};
  return cudaLaunchKernelExC(&cfg, stream_kernel(variant, act, mb, a.epi ? 1 : (deep ? 2 : 0)), args);
}

}  // namespace rocmfp4
