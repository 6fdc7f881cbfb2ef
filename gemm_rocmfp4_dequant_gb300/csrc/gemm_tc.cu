// W4A16 GEMM on sm_103a tensor cores:  Y[M][N] = X[M][K] . W[N][K]^T, with X
// fp16 or bf16 (row-major), W packed ROCmFP4 blocks (dual or single-scale),
// Y fp32 (row-major, overwritten).
//
// The weight decode follows "Feasibility Report: Porting ROCmFP4 to Atlas",
// section "What is ROCmFP4?" (Block Layout, Codebook10 Value Table, Scale
// Format); common.cuh explains the exact e2m1 / e4m3 conversion route.  Each
// decoded weight is exact in fp16 and in bf16, so every tensor-core product
// is exact; only the fp32 accumulation rounds.
//
// Tiles.  A CTA computes the transposed tile Y^T[n0 .. n0+127][m0 .. m0+NT-1]
// (NT <= 256 tokens) with tcgen05.mma, kind::f16, M = 128 weight rows,
// N = NT, K = 16 per instruction, both operands in shared memory in the
// 128-byte-swizzled K-major layout:
//   A = 64-K slices of the weight tile, decoded into shared memory by the
//       decode warps (one 128-byte row per weight row);
//   B = the matching 64-K slice of X rows m0 .. m0+NT-1, staged by TMA.
// The accumulator's lanes are weight rows, so the epilogue's stores of one
// warp cover 32 consecutive outputs of a row of Y.  CTAs are persistent and
// walk the tiles in a grouped order (a group of token tiles is swept across
// all weight tiles), so a weight tile is fetched from HBM about once per
// group while the group's X stays in L2.
//
// Accumulation chains.  The tensor core adds each 16-deep partial product
// into its fp32 accumulator with a rounding whose error grows with the chain
// length (at K = 17408 one chain leaves a relative L2 error near 1.2e-5).
// K is therefore cut into chains of at most kChainK: chain 0 of a tile
// accumulates in one of the two tensor-memory slots (its base slot), every
// later chain in the other; after each later chain the output warps add the
// other slot into the base slot (fp32, round to nearest).  The base slot
// alternates between consecutive tiles, so the next tile's chain 0 runs in
// the freed slot while the finished tile is still being stored.  The order
// of all additions is fixed, so results are deterministic.
//
// Split tiles (the last wave and a half when the tile count is not a
// multiple of the SM count) are cut by K across consecutive CTAs.  The CTA
// holding a tile's first chunk keeps that part in tensor memory and, after
// its roles end, adds the other parts (written to a workspace) in chunk
// order; such a launch is cooperative because that CTA waits for the others.
//
// Warp roles (512 threads):
//   warp 0       TMA producer of the X slices
//   warp 1       tensor-memory allocation and the MMA issue (one thread)
//   warp 2       TMA producer of raw ROCmFP4 chunks (128 rows x 256 or 512 K)
//   warp 3       idle after set-up
//   warps 4-11   decode: warp w handles rows 32*(w % 4) .. +31 (one thread
//                per row) of the 64-K slices of parity (w - 4) / 4, so two
//                slices are decoded at once
//   warps 12-15  chain folds and the epilogue (tensor-memory lanes 32*(w % 4))
// A stage (X slice + decoded A slice) is released by one tcgen05.commit.
// Every wait is bounded: a warp that gives up records kErrWaitTimeout and
// leaves its loops, and all warps still meet at the final barrier that
// precedes the tensor-memory release.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "kernels.h"

namespace rocmfp4 {
namespace {

constexpr int kTcRows = 128;       // weight rows per tile (MMA M)
constexpr int kSubK = 64;          // K per stage
constexpr int kThreads = 512;
constexpr int kDecWarps = 8;       // warps 4-11
constexpr int kOutThreads = 128;   // warps 12-15
constexpr int kMaxStages = 8;
constexpr int kMaxNT = 256;        // tokens per tile
constexpr int kChainK = 4096;      // longest accumulation chain
constexpr uint32_t kABytes = kTcRows * 128;  // decoded A slice: 128 rows x 64 K x 16 bit
constexpr uint32_t kSmemBudget = 227 * 1024;

template <int V>
struct TcFmt {
  static constexpr int BB = Fmt<V>::BB;
  static constexpr int KR = V == 0 ? 256 : 512;          // K per raw chunk
  static constexpr int RSPAN = KR / 32 * BB;             // raw bytes per row per chunk: 144 / 272
  static constexpr int RW = RSPAN / 4;                   // words per row per chunk
  static constexpr int SUBS = KR / kSubK;                 // 64-K slices per chunk: 4 / 8
  static constexpr int RSTAGES = V == 0 ? 3 : 2;         // raw chunk ring
  static constexpr int RBYTES = kTcRows * RSPAN;         // one raw stage
  static constexpr int EBUF = V == 0 ? 2 : 1;            // epilogue buffers per output warp
};
constexpr uint32_t kEpiBytes = 16 * 32 * 4;  // one epilogue buffer: 16 tokens x 32 outputs, fp32
constexpr uint32_t kFixStageBytes = (kThreads / 32) * 2 * kEpiBytes;  // split fix-up: two buffers per warp
constexpr int kFixWinGroups = 2 * kThreads / 128;  // split fix-up: 16-token groups per window, at most

// Shared- and tensor-memory plan for a token-tile width nt (multiple of 16, <= 256).
struct TcPlan {
  uint32_t xbytes;      // X slice: nt rows of 128 bytes
  uint32_t sbytes;      // one stage: X slice + decoded A slice
  uint32_t stages;      // stage ring depth
  uint32_t off_raw;     // raw ring
  uint32_t off_epi;     // epilogue buffers
  uint32_t off_bar;     // mbarriers
  uint32_t smem;        // dynamic bytes requested (with 1 KB alignment slack)
  uint32_t cstride;     // tensor-memory columns per accumulator slot
  uint32_t tmem_cols;   // tensor-memory allocation: slots R and C
};

RF4_HOSTDEV TcPlan tc_plan(int variant, int nt) {
  TcPlan p;
  p.xbytes = (uint32_t)nt * 128u;
  p.sbytes = p.xbytes + kABytes;
  const uint32_t raw = variant == 0 ? TcFmt<0>::RSTAGES * TcFmt<0>::RBYTES : TcFmt<1>::RSTAGES * TcFmt<1>::RBYTES;
  const uint32_t epi = 4u * kEpiBytes * (variant == 0 ? TcFmt<0>::EBUF : TcFmt<1>::EBUF);
  const uint32_t fixed = raw + epi + 512 + 1024;  // raw ring, epilogue buffers, barriers, alignment slack
  uint32_t s = (kSmemBudget - fixed) / p.sbytes;
  p.stages = s > (uint32_t)kMaxStages ? (uint32_t)kMaxStages : s;
  p.off_raw = p.stages * p.sbytes;
  p.off_epi = p.off_raw + raw;
  p.off_bar = p.off_epi + epi;
  p.smem = p.off_bar + 512 + 1024;
  p.cstride = nt <= 128 ? 128u : 256u;
  p.tmem_cols = 2 * p.cstride;
  // Co-resident CTAs must fit in the SM's 512 tensor-memory columns: a
  // 512-column CTA asks for more than half of the SM's 228 KB of shared
  // memory, a 256-column CTA for more than a third.
  const uint32_t floor_bytes = p.tmem_cols == 512 ? 117u * 1024u : 78u * 1024u;
  if (p.smem < floor_bytes) p.smem = floor_bytes;
  return p;
}

// Tile order: group_m consecutive token tiles are swept across every weight
// tile before the next group starts.
struct Raster {
  int mtiles, ntiles, group_m, nt;
  RF4_DEV void tile(int t, int& m0, int& n0) const {
    const int per_group = group_m * ntiles;
    const int g = t / per_group, in_g = t % per_group;
    const int first = g * group_m;
    const int gsize = min(mtiles - first, group_m);
    m0 = (first + in_g % gsize) * nt;
    n0 = (in_g / gsize) * kTcRows;
  }
};

// Work items.  Tiles 0 .. dp_tiles-1 are dealt out whole, round robin (full
// waves of the grid).  The remaining tiles form the split region: its
// tiles x nch raw chunks are numbered tile-major and cut into gridDim.x
// contiguous ranges of near-equal length, one per CTA, so every SM gets the
// same amount of work however the tile count falls against the SM count.
// A range yields one item per tile it touches: (tile, chunk range).
struct Sched {
  int dp_tiles;  // tiles dealt out whole
  int nch;       // raw chunks per tile (K / KR)
  int64_t usk;   // chunks of the split region
  RF4_DEV int64_t start(int b) const { return (int64_t)b * usk / gridDim.x; }
  // The CTA whose range holds chunk u: the largest b with start(b) <= u.
  RF4_DEV int owner(int64_t u) const { return (int)(((u + 1) * (int64_t)gridDim.x - 1) / usk); }
};

struct Item {
  int t, cb, ce;  // tile and its raw chunks [cb, ce)
};

struct ItemIter {
  int next_dp;
  int64_t u, uend;
  RF4_DEV explicit ItemIter(const Sched& s)
      : next_dp((int)blockIdx.x), u(s.start((int)blockIdx.x)), uend(s.start((int)blockIdx.x + 1)) {}
  RF4_DEV bool next(const Sched& s, Item& it) {
    if (next_dp < s.dp_tiles) {
      it.t = next_dp;
      it.cb = 0;
      it.ce = s.nch;
      next_dp += (int)gridDim.x;
      return true;
    }
    if (u >= uend) return false;
    const int64_t tr = u / s.nch;
    it.t = s.dp_tiles + (int)tr;
    it.cb = (int)(u - tr * s.nch);
    const int64_t left = uend - u;
    it.ce = left < (int64_t)(s.nch - it.cb) ? it.cb + (int)left : s.nch;
    u += it.ce - it.cb;
    return true;
  }
};

constexpr int kSubsPerChain = kChainK / kSubK;
constexpr size_t kSlotFloats = (size_t)kTcRows * kMaxNT;  // one partial tile in the split workspace

RF4_DEV void epi_bar_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kOutThreads) : "memory"); }

// One partial tile in the split workspace: [token group g][quad q][row][4],
// token 16 g + 4 q + i of weight row `row` at element i, so that a warp's
// float4 access of one (g, q) covers 512 contiguous bytes.
RF4_DEV size_t part_index(int g, int q, int row) { return (((size_t)g * 4 + q) * kTcRows + row) * 4; }

// The parts of one split tile: part k is CTA (bfirst + k)'s.  Part 0 stays
// in CTA bfirst's tensor memory; part k >= 1 starts CTA (bfirst + k)'s range
// and is in that CTA's workspace slot.
struct Parts {
  const float* ws;
  int bfirst, nparts;
  RF4_DEV const float* slot(int k) const { return ws + (size_t)(bfirst + k) * kSlotFloats; }
};

// Waits (bounded: about two seconds of SM clock, acquire) until a split
// tile's count of written parts reaches `need`; false if it gave up.  The
// writers wait on nothing of the waiting CTA's, and a grid with split tiles
// is launched cooperatively, so every writer is resident.
RF4_DEV bool wait_parts_written(uint32_t* cnt, uint32_t need) {
  const long long t0 = clock64();
  for (;;) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(cnt) : "memory");
    if (v >= need) return true;
    if (clock64() - t0 > (1ll << 32)) return false;
    __nanosleep(32);
  }
}

RF4_DEV Parts tile_parts(const Sched& sc, const float* ws, int t) {
  const int64_t t0 = (int64_t)(t - sc.dp_tiles) * sc.nch;
  Parts p;
  p.ws = ws;
  p.bfirst = sc.owner(t0);
  p.nparts = sc.owner(t0 + sc.nch - 1) - p.bfirst + 1;
  return p;
}

RF4_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
RF4_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

RF4_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Bounded wait whose outcome is the same for the whole warp (the tcgen05
// loads and stores that follow are warp-collective).
RF4_DEV bool warp_wait(uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity));
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzle layout: rows of 128 bytes, 8-row groups 1024 bytes apart.
RF4_DEV uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16;              // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;    // stride byte offset: next 8-row group
  d |= (uint64_t)1 << 46;              // descriptor version
  d |= (uint64_t)2 << 61;              // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp32 accumulator, A and B both fp16
// (act 0) or both bf16 (act 1), both K-major, N = nt, M = 128.
RF4_DEV uint32_t instr_desc(int act, int nt) {
  return (1u << 4) | ((uint32_t)act << 7) | ((uint32_t)act << 10) | ((uint32_t)(nt >> 3) << 17) |
         ((uint32_t)(kTcRows >> 4) << 24);
}

// D[tmem] (+)= A[smem] . B[smem]^T
RF4_DEV void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

RF4_DEV void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// Byte `pos` of a word array as an E2M1 pair (pos is a constant after unrolling).
template <int NW>
RF4_DEV uint32_t e2m1_at(const uint32_t (&w)[NW], int pos) {
  const uint32_t word = w[pos >> 2];
  switch (pos & 3) {
    case 0: return e2m1x2<0>(word);
    case 1: return e2m1x2<1>(word);
    case 2: return e2m1x2<2>(word);
    default: return e2m1x2<3>(word);
  }
}

// Scale pair of the block whose scale byte(s) start at byte `pos`: the two
// E4M3 values of a dual block, or the one of a single-scale block twice.
template <int V, int NW>
RF4_DEV uint32_t scales_at(const uint32_t (&w)[NW], int pos) {
  if constexpr (V == 0) {
    return (pos & 2) ? e4m3x2<1>(w[pos >> 2]) : e4m3x2<0>(w[pos >> 2]);  // dual scales sit at even offsets
  } else {
    return e4m3x2<0>(__byte_perm(w[pos >> 2], 0u, (uint32_t)(pos & 3) * 0x11u));
  }
}

RF4_DEV uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Decode the block starting at byte `pos` of w into 16 packed words:
// out[i] = (w_2i, w_2i+1), out[8 + i] = (w_2i+16, w_2i+17), i = 0..7.
template <int V, int ACT, int NW>
RF4_DEV void decode_block(const uint32_t (&w)[NW], int pos, uint32_t (&out)[16]) {
  const uint32_t s2 = scales_at<V>(w, pos + 16);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    // byte j holds (w_j, w_j+16); the products are exact in fp16
    const uint32_t a = hmul2(clamp5(e2m1_at(w, pos + 2 * i)), s2);
    const uint32_t b = hmul2(clamp5(e2m1_at(w, pos + 2 * i + 1)), s2);
    if constexpr (ACT == 0) {
      out[i] = __byte_perm(a, b, 0x5410);
      out[8 + i] = __byte_perm(a, b, 0x7632);
    } else {
      const __half2 ha = *reinterpret_cast<const __half2*>(&a);
      const __half2 hb = *reinterpret_cast<const __half2*>(&b);
      out[i] = pack_bf16x2(__low2float(ha), __low2float(hb));
      out[8 + i] = pack_bf16x2(__high2float(ha), __high2float(hb));
    }
  }
}

RF4_DEV void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

RF4_DEV void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// AND of v over the 128 output threads (named barrier 1).
RF4_DEV bool epi_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kOutThreads)
      : "memory");
  return r != 0;
}

// Stores of one output warp: 16 tokens x its 32 outputs (tensor-memory lanes)
// of Y, through shared memory and a TMA tensor store when Y's rows are
// 16-byte aligned (rows past M and columns past N are not written), else
// plain stores.
template <int EBUF>
struct Emit {
  uint8_t* ebuf;  // EBUF buffers of kEpiBytes
  int ebi;
  int quarter, lane, tma_y;
  const CUtensorMap* tmy;
  float* Y;
  int M, N;
  RF4_DEV void store(const uint32_t (&a)[16], int m, int n0) {
    if (tma_y) {
      uint8_t* buf = ebuf + (uint32_t)ebi * kEpiBytes;
      if (lane == 0) bulk_wait_group_read<EBUF - 1>();  // the buffer's previous store has read it
      __syncwarp();
      float* fb = reinterpret_cast<float*>(buf);
#pragma unroll
      for (int j = 0; j < 16; ++j) fb[j * 32 + lane] = __uint_as_float(a[j]);
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        if (n0 + quarter * 32 < N && m < M) tma_store_2d(tmy, n0 + quarter * 32, m, smem_addr(buf));
        bulk_commit_group();
      }
      ebi = ebi + 1 == EBUF ? 0 : ebi + 1;
    } else {
      const int n = n0 + quarter * 32 + lane;
      if (n < N) {
        float* y = Y + (size_t)m * N + n;
        const int mlim = M - m;
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (j < mlim) y[(size_t)j * N] = __uint_as_float(a[j]);
      }
    }
  }
};

// Ring position: stage index and the parity of its current use.
struct Ring {
  uint32_t stage = 0;
  uint32_t phase = 0;
  RF4_DEV void next(uint32_t n) {
    if (++stage == n) {
      stage = 0;
      phase ^= 1u;
    }
  }
};

struct Bars {
  uint64_t* full;     // [stages] X bytes + one arrival per decode warp
  uint64_t* empty;    // [stages] MMA commit
  uint64_t* rfull;    // [raw stages] TMA bytes
  uint64_t* rempty;   // [raw stages] one arrival per decode warp
  uint64_t* cfull;    // [2] chain finished in accumulator slot 0 / 1 (MMA commit)
  uint64_t* sfree;    // [2] accumulator slot consumed: folded or read out (output warps)
  uint64_t* fixbar;   // [2] split fix-up: bulk copies of the parts into buffer 0 / 1 (TMA bytes)
};

// Slice S (two blocks, 64 K) of the raw chunk, for this thread's weight row,
// into its 128-byte row of the A slice (16-byte chunk c stored at c ^ (row % 8)).
template <int V, int ACT, int S>
RF4_DEV void decode_slice_to_smem(const uint8_t* rrow, uint8_t* arow, int row) {
  using F = TcFmt<V>;
  constexpr int lo = 2 * S * F::BB;  // first byte of the slice's two blocks in the chunk row
  constexpr int a0 = lo / 16 * 16;   // 16-byte aligned 48-byte window
  static_assert(a0 + 48 <= F::RSPAN && lo - a0 + 2 * F::BB <= 48, "slice window");
  uint32_t w[12];
  const uint4* src = reinterpret_cast<const uint4*>(rrow + a0);
#pragma unroll
  for (int q = 0; q < 3; ++q) {
    const uint4 v = src[q];
    w[4 * q] = v.x;
    w[4 * q + 1] = v.y;
    w[4 * q + 2] = v.z;
    w[4 * q + 3] = v.w;
  }
  uint32_t out0[16], out1[16];
  decode_block<V, ACT>(w, lo - a0, out0);
  decode_block<V, ACT>(w, lo - a0 + F::BB, out1);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t* o = c < 4 ? out0 + 4 * c : out1 + 4 * (c - 4);
    *reinterpret_cast<uint4*>(arow + ((c ^ (row & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// The slices of parity HALF of one raw chunk (the other decode set takes the
// rest); false if a wait gave up.  The ring advances over every slice.
template <int V, int ACT, int HALF, int S = HALF>
RF4_DEV bool decode_chunk(const uint8_t* rrow, uint8_t* abase, uint32_t sbytes, uint32_t stages, int row, int lane,
                          Ring& ring, const Bars& b, uint32_t rempty_bar) {
  if constexpr (S >= TcFmt<V>::SUBS) {
    return true;
  } else {
    // The stage is free once the MMAs of its previous use have completed (on
    // the first pass the wait is for the phase before a fresh barrier's
    // first one, which counts as complete).
    if (!warp_wait(smem_addr(&b.empty[ring.stage]), ring.phase ^ 1u)) return false;
    uint8_t* arow = abase + (size_t)ring.stage * sbytes + (size_t)row * 128;
    decode_slice_to_smem<V, ACT, S>(rrow, arow, row);
    if constexpr (S + 2 >= TcFmt<V>::SUBS) {
      __syncwarp();
      if (lane == 0) mbar_arrive(rempty_bar);  // the warp's last read of the chunk
    }
    fence_proxy_async();  // make the generic-proxy stores visible to the tensor core
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&b.full[ring.stage]));
    ring.next(stages);
    ring.next(stages);
    return decode_chunk<V, ACT, HALF, S + 2>(rrow, abase, sbytes, stages, row, lane, ring, b, rempty_bar);
  }
}

template <int V, int ACT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
                   const __grid_constant__ CUtensorMap tmy, int tma_y, float* __restrict__ Y, int M, int N, int K,
                   int nt, int mtiles, int ntiles, int group_m, Sched sched, float* __restrict__ ws,
                   uint32_t* __restrict__ tcnt, uint32_t* __restrict__ err) {
  using F = TcFmt<V>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const TcPlan plan = tc_plan(V, nt);
  const uint32_t S = plan.stages;
  uint8_t* stage0 = smem;                 // stage s: X slice at s*sbytes, A slice right after it
  uint8_t* rs = smem + plan.off_raw;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + plan.off_bar);
  Bars b;
  b.full = bar;
  b.empty = b.full + kMaxStages;
  b.rfull = b.empty + kMaxStages;
  b.rempty = b.rfull + F::RSTAGES;
  b.cfull = b.rempty + F::RSTAGES;
  b.sfree = b.cfull + 2;
  b.fixbar = b.sfree + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(b.fixbar + 2);
  // The split tile whose first part is this CTA's final item (at most one),
  // summed by all threads after the roles end: {count, then (tile, m0, n0,
  // own accumulator slot) per tile}.
  volatile int* fix = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* wait_flag = fix + 12;  // the fix-up's wait for written parts

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Raster raster{mtiles, ntiles, group_m, nt};

  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < S; ++i) {
      mbar_init(smem_addr(&b.full[i]), 1 + kDecWarps / 2);  // X bytes + the 4 warps of one decode set
      mbar_init(smem_addr(&b.empty[i]), 1);
    }
    for (int i = 0; i < F::RSTAGES; ++i) {
      mbar_init(smem_addr(&b.rfull[i]), 1);
      mbar_init(smem_addr(&b.rempty[i]), kDecWarps);
    }
    mbar_init(smem_addr(&b.cfull[0]), 1);
    mbar_init(smem_addr(&b.cfull[1]), 1);
    mbar_init(smem_addr(&b.sfree[0]), kOutThreads);
    mbar_init(smem_addr(&b.sfree[1]), kOutThreads);
    mbar_init(smem_addr(&b.fixbar[0]), 1);
    mbar_init(smem_addr(&b.fixbar[1]), 1);
    fix[0] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(plan.tmem_cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---- X producer ----
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmx)) : "memory");
      Ring r;
      bool ok = true;
      ItemIter it(sched);
      Item w;
      while (ok && it.next(sched, w)) {
        int m0, n0;
        raster.tile(w.t, m0, n0);
        for (int ks = w.cb * F::SUBS; ks < w.ce * F::SUBS; ++ks, r.next(S)) {
          if (!mbar_wait_bounded(smem_addr(&b.empty[r.stage]), r.phase ^ 1u)) {
            ok = false;
            break;
          }
          const uint32_t full = smem_addr(&b.full[r.stage]);
          mbar_arrive_expect_tx(full, plan.xbytes);
          tma_load_2d(smem_addr(stage0 + (size_t)r.stage * plan.sbytes), &tmx, ks * kSubK, m0, full);
        }
      }
      if (!ok) atomicOr(err, kErrWaitTimeout);
    }
  } else if (warp == 2) {
    // ---- raw weight producer ----
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmw)) : "memory");
      Ring r;
      bool ok = true;
      ItemIter it(sched);
      Item w;
      while (ok && it.next(sched, w)) {
        int m0, n0;
        raster.tile(w.t, m0, n0);
        for (int rc = w.cb; rc < w.ce; ++rc, r.next(F::RSTAGES)) {
          if (!mbar_wait_bounded(smem_addr(&b.rempty[r.stage]), r.phase ^ 1u)) {
            ok = false;
            break;
          }
          const uint32_t full = smem_addr(&b.rfull[r.stage]);
          mbar_arrive_expect_tx(full, F::RBYTES);
          tma_load_2d(smem_addr(rs + (size_t)r.stage * F::RBYTES), &tmw, rc * F::RW, n0, full);
        }
      }
      if (!ok) atomicOr(err, kErrWaitTimeout);
    }
  } else if (warp == 1) {
    // ---- MMA issue ----
    if (lane == 0) {
      const uint32_t idesc = instr_desc(ACT, nt);
      const uint64_t xdesc0 = smem_desc_sw128(smem_addr(stage0));
      const uint64_t adesc0 = smem_desc_sw128(smem_addr(stage0 + plan.xbytes));
      Ring r;
      uint32_t uses0 = 0, uses1 = 0;  // chains written into each accumulator slot so far
      bool ok = true;
      ItemIter it(sched);
      Item w;
      for (int item = 0; ok && it.next(sched, w); ++item) {
        const int s0 = w.cb * F::SUBS, nsub = (w.ce - w.cb) * F::SUBS;
        const int nchains = (nsub + kSubsPerChain - 1) / kSubsPerChain;
        const int base = item & 1;  // chain 0 of the item; later chains use the other slot
        int ks = s0;
        for (int c = 0; c < nchains && ok; ++c) {
          const int kend = s0 + (int)((int64_t)(c + 1) * nsub / nchains);
          // a slot takes a new chain once the output warps have consumed its previous one
          const int sl = c == 0 ? base : base ^ 1;
          const uint32_t un = sl ? uses1 : uses0;
          if (un > 0 && !mbar_wait_bounded(smem_addr(&b.sfree[sl]), (un - 1) & 1u)) {
            ok = false;
            break;
          }
          if (sl) ++uses1; else ++uses0;
          tc_fence_after();
          const uint32_t d = tmem + (uint32_t)sl * plan.cstride;
          for (int k0 = ks; ks < kend; ++ks, r.next(S)) {
            if (!mbar_wait_bounded(smem_addr(&b.full[r.stage]), r.phase)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t off = (uint64_t)((r.stage * plan.sbytes) >> 4);
#pragma unroll
            for (int k = 0; k < kSubK / 16; ++k)
              mma_ss(d, adesc0 + off + 2 * k, xdesc0 + off + 2 * k, idesc, (ks != k0) || (k != 0));
            mma_commit(smem_addr(&b.empty[r.stage]));
          }
          // The output warps act on every chain but the first of several.
          if (ok && (c > 0 || nchains == 1)) mma_commit(smem_addr(&b.cfull[sl]));
        }
      }
      if (!ok) atomicOr(err, kErrWaitTimeout);
    }
  } else if (warp >= 4 && warp < 12) {
    // ---- decode ----
    const int quarter = warp & 3;
    const int half = (warp - 4) >> 2;      // decode set: slices of this parity
    const int row = quarter * 32 + lane;   // weight row of the tile
    uint8_t* abase = stage0 + plan.xbytes;
    Ring rr, ring;
    if (half) ring.next(S);
    bool ok = true;
    ItemIter it(sched);
    Item w;
    while (ok && it.next(sched, w)) {
      for (int rc = w.cb; rc < w.ce; ++rc, rr.next(F::RSTAGES)) {
        if (!warp_wait(smem_addr(&b.rfull[rr.stage]), rr.phase)) {
          ok = false;
          break;
        }
        const uint8_t* rrow = rs + (size_t)rr.stage * F::RBYTES + (size_t)row * F::RSPAN;
        const uint32_t re = smem_addr(&b.rempty[rr.stage]);
        ok = half == 0 ? decode_chunk<V, ACT, 0>(rrow, abase, plan.sbytes, S, row, lane, ring, b, re)
                       : decode_chunk<V, ACT, 1>(rrow, abase, plan.sbytes, S, row, lane, ring, b, re);
        if (!ok) break;
      }
    }
    if (!ok && lane == 0) atomicOr(err, kErrWaitTimeout);
  } else if (warp >= 12) {
    // ---- chain folds and epilogue ----
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;  // tensor-memory lane = weight row of the tile
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    Emit<F::EBUF> out{smem + plan.off_epi + (uint32_t)quarter * F::EBUF * kEpiBytes, 0, quarter, lane, tma_y, &tmy, Y,
                      M, N};
    uint32_t n_cfull0 = 0, n_cfull1 = 0;  // chain completions awaited per slot
    bool ok = true;
    ItemIter it(sched);
    Item w;
    for (int item = 0; ok && it.next(sched, w); ++item) {
      int m0, n0;
      raster.tile(w.t, m0, n0);
      const int nsub = (w.ce - w.cb) * F::SUBS;
      const int nchains = (nsub + kSubsPerChain - 1) / kSubsPerChain;
      // chain 0 accumulates in the item's base slot, later chains in the other
      const int base = item & 1;
      const uint32_t slot_b = tmem + lane_off + (uint32_t)base * plan.cstride;
      const uint32_t slot_o = tmem + lane_off + (uint32_t)(base ^ 1) * plan.cstride;
      const bool whole = w.cb == 0 && w.ce == sched.nch;
      // A split tile's first part (chunk 0 on) ends its CTA's range, so it is
      // that CTA's final item: the CTA keeps it in tensor memory and sums
      // the tile once its roles have ended.  Every other part starts its
      // CTA's range and goes to that CTA's workspace slot.
      const bool keep = !whole && w.cb == 0;
      float* part = ws + (size_t)blockIdx.x * kSlotFloats;
      for (int c = nchains > 1 ? 1 : 0; c < nchains; ++c) {  // chain 0 of several stays in the base slot
        // the four output warps leave together, so their named barriers stay matched
        const int sl = c == 0 ? base : base ^ 1;
        const uint32_t nc = sl ? n_cfull1++ : n_cfull0++;
        if (!(ok = epi_all(warp_wait(smem_addr(&b.cfull[sl]), nc & 1u)))) break;
        tc_fence_after();
        if (nchains > 1) {
          // base += other (fp32, round to nearest); the other slot is then
          // free: for the next chain, or, after the last one, for the next
          // item's chain 0 while this item's result is still being stored
#pragma unroll 1
          for (int c0 = 0; c0 < nt; c0 += 16) {
            uint32_t a[16], v[16];
            tmem_ld16(slot_b + (uint32_t)c0, a);
            tmem_ld16(slot_o + (uint32_t)c0, v);
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
            for (int j = 0; j < 16; ++j) a[j] = __float_as_uint(__uint_as_float(a[j]) + __uint_as_float(v[j]));
            tmem_st16(slot_b + (uint32_t)c0, a);
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          tc_fence_before();
          mbar_arrive(smem_addr(&b.sfree[base ^ 1]));
          if (c + 1 < nchains) continue;
        }
        if (keep) {
          if (row == 0) {
            const int i = fix[0];
            fix[1 + 4 * i] = w.t;
            fix[2 + 4 * i] = m0;
            fix[3 + 4 * i] = n0;
            fix[4 + 4 * i] = base;  // part 0 of the tile: this CTA's, in this slot
            fix[0] = i + 1;
          }
          break;
        }
        // the base slot holds the item's sum: 16 tokens at a time to Y or to the workspace
#pragma unroll 1
        for (int c0 = 0; c0 < nt; c0 += 16) {
          uint32_t a[16];
          tmem_ld16(slot_b + (uint32_t)c0, a);
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
          if (c0 + 16 >= nt) {
            tc_fence_before();
            mbar_arrive(smem_addr(&b.sfree[base]));  // read out: the slot may take a new chain
          }
          if (whole) {
            out.store(a, m0 + c0, n0);
          } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              __stcg(reinterpret_cast<float4*>(part + part_index(c0 / 16, q, row)),
                     make_float4(__uint_as_float(a[4 * q]), __uint_as_float(a[4 * q + 1]),
                                 __uint_as_float(a[4 * q + 2]), __uint_as_float(a[4 * q + 3])));
          }
        }
      }
      if (!ok || whole || keep) continue;
      // Split tile, part written: count it for the tile's first CTA, which
      // waits for the count after its own roles have ended.  A part is
      // written before its CTA waits on anything of another CTA's, and the
      // owners of later parts have higher indices, so no wait is circular.
      epi_bar_sync();  // every output thread's part stores precede the count
      if (row == 0) {
        __threadfence();  // this CTA's part is visible before the count
        atomicAdd(&tcnt[w.t - sched.dp_tiles], 1u);
      }
    }
    if (lane == 0) bulk_wait_group_all();  // the stores have left shared memory and completed
    if (!ok && lane == 0) atomicOr(err, kErrWaitTimeout);
  }

  tc_fence_before();
  __syncthreads();
  // ---- split fix-up: all threads; the stage and raw rings are free ----
  // The recorded tile's part 0 is in this CTA's tensor memory.  Wait until
  // the other parts are written, bring them into shared memory by bulk
  // copies, window by window into two alternating buffers (the copies of
  // the next window overlap the sums of this one), add the parts in chunk
  // order and store the tile.  Tensor memory is released afterwards.
  tc_fence_after();
  const int nfix = fix[0];
  uint32_t fix_phase = 0;  // bit i: parity of fixbar[i]
  bool fix_ok = true;
  const uint32_t tlane = tmem + ((uint32_t)(32 * (warp & 3)) << 16);  // this warp's tensor-memory lanes
  // Every warp stages its 16 x 32 output blocks for tensor stores in two
  // buffers of its own, just below the epilogue buffers.
  Emit<2> fout{smem + plan.off_epi - kFixStageBytes + (uint32_t)warp * 2 * kEpiBytes, 0, warp & 3, lane, tma_y, &tmy,
               Y, M, N};
#pragma unroll 1
  for (int f = 0; f < nfix; ++f) {
    const int t = fix[1 + 4 * f], m0 = fix[2 + 4 * f], n0 = fix[3 + 4 * f];
    const uint32_t own_slot = tlane + (uint32_t)fix[4 + 4 * f] * plan.cstride;
    const Parts parts = tile_parts(sched, ws, t);
    const int ncopy = parts.nparts - 1;
    if (threadIdx.x == 0) {
      uint32_t* cnt = &tcnt[t - sched.dp_tiles];
      const bool okw = wait_parts_written(cnt, (uint32_t)ncopy);
      if (okw) atomicExch(cnt, 0u);  // every contributor is done with it: ready for the next launch
      *wait_flag = okw ? 1 : 0;
    }
    __syncthreads();
    if (*wait_flag == 0) {
      fix_ok = false;
      __syncthreads();  // every thread has read the flag before thread 0 writes it again
      continue;
    }
    const int groups = nt / 16;
    constexpr uint32_t kGroupBytes = kTcRows * 16 * 4;  // one part, 16 tokens
    // token groups per window: two windows of every copied part fit in the
    // rings below the store staging buffers; at most kFixWinGroups, so that
    // a thread holds at most two (row, group) pairs of a window
    const uint32_t half_area = ((plan.off_epi - kFixStageBytes) / 2) & ~15u;
    const int win = min(min(groups, kFixWinGroups), (int)(half_area / ((uint32_t)max(ncopy, 1) * kGroupBytes)));
    const bool from_ws = win == 0;  // too many parts for shared memory: read them in place
    const int step = from_ws ? 1 : win;
    const int nwin = (groups + step - 1) / step;
    // window w of the copied parts: part k (1..) at buffer (w & 1), slot k - 1
    auto issue = [&](int w) {
      const int g0 = w * step, gw = min(step, groups - g0);
      const uint32_t pbytes = (uint32_t)gw * kGroupBytes;
      uint8_t* buf = smem + (size_t)(w & 1) * half_area;
      const uint32_t bar = smem_addr(&b.fixbar[w & 1]);
      // the buffer's earlier generic-proxy accesses, and the parts acquired
      // through the counter, come before the bulk copies
      asm volatile("fence.proxy.async;" ::: "memory");
      mbar_arrive_expect_tx(bar, pbytes * (uint32_t)ncopy);
      for (int k = 1; k < parts.nparts; ++k)
        bulk_g2s(smem_addr(buf + (size_t)(k - 1) * pbytes), parts.slot(k) + (size_t)g0 * kTcRows * 16, pbytes, bar);
    };
    if (!from_ws && threadIdx.x == 0) issue(0);
#pragma unroll 1
    for (int w = 0; w < nwin; ++w) {
      const int g0 = w * step, gw = min(step, groups - g0);
      const uint32_t pbytes = (uint32_t)gw * kGroupBytes;
      const uint8_t* buf = smem + (size_t)(w & 1) * half_area;
      if (!from_ws && threadIdx.x == 0 && w + 1 < nwin) issue(w + 1);
      // part 0 of this thread's (row, group) pairs, from tensor memory, while
      // the copies land: a warp's lanes are 32 rows of its tensor-memory lane
      // quarter and share one group, as the tensor-memory loads need
      uint32_t own[2][16];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int pi = threadIdx.x + i * kThreads;
        if (pi < kTcRows * gw) tmem_ld16(own_slot + (uint32_t)(16 * (g0 + pi / kTcRows)), own[i]);
      }
      asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
      if (!from_ws) {
        fix_ok = mbar_wait_bounded(smem_addr(&b.fixbar[w & 1]), (fix_phase >> (w & 1)) & 1u) && fix_ok;
        fix_phase ^= 1u << (w & 1);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int pi = threadIdx.x + i * kThreads;
        if (pi >= kTcRows * gw) break;
        const int row = pi % kTcRows, gl = pi / kTcRows, g = g0 + gl;
        float4 s4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          s4[q] = make_float4(__uint_as_float(own[i][4 * q]), __uint_as_float(own[i][4 * q + 1]),
                              __uint_as_float(own[i][4 * q + 2]), __uint_as_float(own[i][4 * q + 3]));
#pragma unroll 1
        for (int k = 1; k < parts.nparts; ++k) {
          float4 v4[4];
          if (from_ws) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              v4[q] = __ldcg(reinterpret_cast<const float4*>(parts.slot(k) + part_index(g, q, row)));
          } else {
            const float4* src =
                reinterpret_cast<const float4*>(buf + (size_t)(k - 1) * pbytes) + (size_t)gl * 4 * kTcRows + row;
#pragma unroll
            for (int q = 0; q < 4; ++q) v4[q] = src[q * kTcRows];
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            s4[q].x += v4[q].x;
            s4[q].y += v4[q].y;
            s4[q].z += v4[q].z;
            s4[q].w += v4[q].w;
          }
        }
        const uint32_t a[16] = {__float_as_uint(s4[0].x), __float_as_uint(s4[0].y), __float_as_uint(s4[0].z),
                                __float_as_uint(s4[0].w), __float_as_uint(s4[1].x), __float_as_uint(s4[1].y),
                                __float_as_uint(s4[1].z), __float_as_uint(s4[1].w), __float_as_uint(s4[2].x),
                                __float_as_uint(s4[2].y), __float_as_uint(s4[2].z), __float_as_uint(s4[2].w),
                                __float_as_uint(s4[3].x), __float_as_uint(s4[3].y), __float_as_uint(s4[3].z),
                                __float_as_uint(s4[3].w)};
        fout.store(a, m0 + 16 * g, n0);
      }
      __syncthreads();  // the window is consumed before copies overwrite its buffer
    }
  }
  if (lane == 0) bulk_wait_group_all();  // the fix-up's stores have completed
  if (!fix_ok) atomicOr(err, kErrWaitTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(plan.tmem_cols));
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

const void* tc_kernel(int v, int act) {
  if (v == 0) return act == 0 ? (const void*)&gemm_tc_kernel<0, 0> : (const void*)&gemm_tc_kernel<0, 1>;
  return act == 0 ? (const void*)&gemm_tc_kernel<1, 0> : (const void*)&gemm_tc_kernel<1, 1>;
}

// Token-tile width: the fewest tiles of at most kMaxNT tokens, balanced, rounded up to 16.
int tc_token_tile(int64_t M) {
  const int64_t tiles = (M + kMaxNT - 1) / kMaxNT;
  const int64_t per = (M + tiles - 1) / tiles;
  return (int)((per + 15) / 16 * 16);
}

int g_sms = 0;

}  // namespace

int tc_k_multiple(int variant) { return variant == 0 ? TcFmt<0>::KR : TcFmt<1>::KR; }
size_t tc_ws_floats(int sms) { return (size_t)sms * kSlotFloats; }
size_t tc_cnt_words(int sms) { return 2 * (size_t)sms; }

cudaError_t tc_prepare() {
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorSymbolNotFound;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&g_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  for (int v = 0; v < 2; ++v)
    for (int a = 0; a < 2; ++a) {
      e = cudaFuncSetAttribute(tc_kernel(v, a), cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBudget);
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}

cudaError_t launch_gemm_tc(int variant, int act, const TcArgs& a, cudaStream_t s) {
  if (!g_encode || g_sms <= 0) return cudaErrorInitializationError;
  const int nt = tc_token_tile(a.M);
  const int64_t mtiles = (a.M + nt - 1) / nt, ntiles = (a.N + kTcRows - 1) / kTcRows;
  if (mtiles * ntiles >= (1LL << 31)) return cudaErrorInvalidConfiguration;
  CUtensorMap tmx, tmw;
  {
    cuuint64_t dims[2] = {(cuuint64_t)a.K, (cuuint64_t)a.M};
    cuuint64_t strides[1] = {(cuuint64_t)a.K * 2};
    cuuint32_t box[2] = {(cuuint32_t)kSubK, (cuuint32_t)nt};
    cuuint32_t es[2] = {1, 1};
    CUresult r = g_encode(&tmx, act == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<uint16_t*>(a.X), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  {
    const int rw = variant == 0 ? TcFmt<0>::RW : TcFmt<1>::RW;
    cuuint64_t dims[2] = {(cuuint64_t)(a.row_bytes / 4), (cuuint64_t)a.N};
    cuuint64_t strides[1] = {(cuuint64_t)a.row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)rw, (cuuint32_t)kTcRows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = g_encode(&tmw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint8_t*>(a.W), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  // Y through TMA when its rows are 16-byte aligned, else plain stores.
  CUtensorMap tmy;
  memset(&tmy, 0, sizeof(tmy));
  int tma_y = 0;
  if (a.N % 4 == 0 && (reinterpret_cast<uintptr_t>(a.Y) & 15u) == 0) {
    cuuint64_t dims[2] = {(cuuint64_t)a.N, (cuuint64_t)a.M};
    cuuint64_t strides[1] = {(cuuint64_t)a.N * 4};
    cuuint32_t box[2] = {32u, 16u};
    cuuint32_t es[2] = {1, 1};
    CUresult r = g_encode(&tmy, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.Y, dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    tma_y = 1;
  }
  const TcPlan plan = tc_plan(variant, nt);
  const int64_t tiles = mtiles * ntiles;
  const int64_t nch = a.K / tc_k_multiple(variant);
  // Whole tiles in full waves of the grid; when the tile count is not a
  // multiple of the SM count, the last wave and a half (or, below one wave,
  // every tile) are split by K so that each SM gets the same number of raw
  // chunks, but no fewer than about 1024 K each.
  const int64_t min_chunks = 1024 / tc_k_multiple(variant);
  Sched sched{(int)tiles, (int)nch, 0};
  int64_t grid = tiles < g_sms ? tiles : g_sms;
  if (tiles % g_sms != 0 && nch >= 2 && a.ws && a.cnt) {
    if (tiles > g_sms) {
      sched.dp_tiles = (int)((tiles / g_sms - 1) * g_sms);
      sched.usk = (tiles - sched.dp_tiles) * nch;
      grid = g_sms;
    } else {
      const int64_t g = std::min<int64_t>(g_sms, tiles * nch / min_chunks);
      if (g > tiles) {
        sched.dp_tiles = 0;
        sched.usk = tiles * nch;
        grid = g;
      }
    }
  }
  float* Y = a.Y;
  float* ws = a.ws;
  uint32_t* tcnt = a.cnt;
  int M = (int)a.M, N = (int)a.N, K = (int)a.K, ntv = nt, mt = (int)mtiles, ntl = (int)ntiles, gm = 8;
  uint32_t* err = a.err;
  void* args[] = {&tmx, &tmw, &tmy, &tma_y, &Y, &M, &N, &K, &ntv, &mt, &ntl, &gm, &sched, &ws, &tcnt, &err};
  // With split tiles the CTA that completes a tile waits for the others'
  // parts: a cooperative launch keeps every CTA resident at once.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = sched.usk > 0 ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, tc_kernel(variant, act), args);
}

}  // namespace rocmfp4
