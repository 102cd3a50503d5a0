// conv_gemm.cuh - implicit-GEMM convolution kernels on the 5th-generation
// tensor cores (tcgen05, accumulators in TMEM).
//
// The three contractions of the conv2d training step (rl-tools
// "operations_generic.h", `forward` Phase 1 and the two scatter updates of
// `backward_full`) are run as GEMMs without materialising im2col:
//   fprop  D[pix][oc]  = sum_k A[pix][k] B[oc][k],  k = (kh,kw,ic),
//          A gathered from X, B = W [OC][KH*KW*IC]
//   dgrad  D[ipix][ic] = sum_k A[ipix][k] B[ic][k], k = (tap,oc) of one
//          stride phase, A gathered from d_conv, B = phase-packed W^T
//   wgrad  D[k][oc]    = sum_pix A[k][pix] B[oc][pix] over a split of the
//          pixels; fp32 partials per split, reduced afterwards.
//
// One persistent CTA per SM (grid = #SMs), 10 warps:
//   warp 0      TMA producer of the B operand (one elected lane)
//   warp 1      TMEM allocator and MMA issuer (one elected lane)
//   warps 2-5   A-operand producers: gather 128-byte rows of NHWC data into
//               128B-swizzled shared memory (cp.async for bf16; load, tf32
//               split and store for fp32)
//   warps 6-9   epilogue: TMEM -> registers -> bias / scale / activation ->
//               global memory
// A ring of `stages` shared-memory stages (full/empty mbarriers) feeds the
// MMA warp; two or more TMEM accumulators (tfull/tempty mbarriers) let the epilogue
// of one tile overlap the main loop of the next.
//
// Precision: BF16 operands accumulate in fp32. FP32 operands run 3xTF32:
// x = hi + lo (both tf32), acc += lo*hi + hi*lo + hi*hi.
#pragma once
#include "ptx.cuh"

namespace c2d {

constexpr int kThreads = 320;
constexpr int kMaxStages = 8;
constexpr int kMaxPhases = 64;
constexpr int kMaxTmaPhases = 4;  // stride phases whose A operand may come by TMA im2col
constexpr int kBM = 128;          // rows of a tile (TMEM lanes)
constexpr int kMaxTmemBufs = 8;   // TMEM accumulators of the fprop / dgrad kernel (512 columns / BN, capped)
constexpr int kLag = 3;           // cp.async groups kept in flight per producer thread (needs >= 4 stages)
constexpr int kTaKb = 4;          // fp32 with A in TMEM: k-blocks of A held in TMEM (hi and lo, 32 columns each)
constexpr int kMaxKps = 2;        // k-blocks per shared-memory stage (TMA paths)

// wait sites recorded in the error word
enum : int { kSiteFull = 1, kSiteEmpty = 2, kSiteTFull = 3, kSiteTEmpty = 4 };

template <int DT>
struct Dt;
template <>
struct Dt<1> {  // bf16
  using T = __nv_bfloat16;
  static constexpr int ES = 2, EC = 8, BKE = 64, UK = 16, NS = 1;
  static constexpr uint32_t FMT = 1;
};
template <>
struct Dt<0> {  // fp32 storage, 3xTF32 arithmetic
  using T = float;
  static constexpr int ES = 4, EC = 4, BKE = 32, UK = 8, NS = 2;
  static constexpr uint32_t FMT = 2;
};

// One stride phase of the row domain. fprop has a single phase; dgrad with
// stride S has S*S phases (input pixels with the same (ih+P) mod S,
// (iw+P) mod S see the same subset of kernel taps).
struct ConvPhase {
  int rows;            // rows of D in this phase: Nimg*Ha*Wa
  int Ha, Wa;          // per-image row grid
  int qh, qw;          // source base: hb = a*rs + qh, wb = b*rs + qw
  int Tw;              // taps along w in this phase
  int K;               // reduction length: taps * Cs
  int num_kb;          // ceil(K / BKE)
  int unit_begin;      // first work unit of this phase
  int b_col;           // first column of this phase in the B matrix
  int oh0, ow0;        // output pixel = (oh0 + a*os, ow0 + b*os)
  int a_lo_h, a_lo_w;  // A by TMA im2col: window corner of row (a, b) = (a*rs + a_lo_h, b*rs + a_lo_w)
  int a_map;           // ... and the index of this phase's im2col map
  int Th, rh, rw;      // dgrad taps: Th rows of taps; the phase's kernel taps are (rh + S t, rw + S u)
  FastDiv div_Wa, div_HaWa, div_Tw;
};

struct ConvGemmParams {
  // B [Nrows][Kcols] K-major: bf16, 2-D boxes of BN rows x 64; fp32 (3xTF32), a 3-D view of the tf32 hi and
  // lo matrices as two planes, boxes of BN rows x 32 x both planes (hi rows then lo rows: one copy per k-block)
  CUtensorMap tmap_b;
  const void* src;        // A source, NHWC [Nimg][Hs][Ws][Cs]
  int Hs, Ws, Cs;
  int rs, tap_sign;       // fprop: rs = stride, taps add; dgrad: rs = 1, taps subtract
  FastDiv div_Cs;
  int num_phases;
  int n_tiles, BN, N;     // N = valid output columns
  int num_units;
  void* out;              // dtype, [pixels][out_ld]
  void* out2;             // optional second output act(v)
  int out_ld, Ho, Wo, os;
  const float* ep_scale;  // optional per-column scale
  const float* ep_shift;  // optional per-column shift
  int act, out_act;       // out = out_act ? act(v) : T(v); out2 = act(T(v))
  float* stats;           // optional batch statistics (count, mean, M2) of v: [m_tile][N][3], or
  int stats_per_cta;      // [blockIdx][N][3] merged over the CTA's tiles (single column tile only)
  int pair;               // CTA pairs (clusters of two, cta_group::2): units are pairs of m-tiles of one phase
                          // (every phase an even count); bf16 with A by TMA; B tiles are BN/2 rows per CTA
  float* rstats;          // optional layer-norm partials of the stored value, one per output pixel,
                          // column tile and epilogue column half (two halves when a_tma, else one):
                          // [pixel][n_tiles][halves][2] = (mean, M2) over the half's columns
  // A operand by TMA im2col (Cs a multiple of one 128-byte channel chunk: 64 bf16 or 32 fp32, one
  // phase): the map walks the row domain; a k-block is (tap, channel chunk) and the tap is the im2col
  // offset, so taps must be non-negative offsets from the window corner (dgrad uses tap-flipped
  // weights for this). fp32: the raw values land in the hi tile and the four producer warps split
  // each stage into tf32 hi / lo before the MMA may read it
  CUtensorMap tmap_a[kMaxTmaPhases];  // one im2col map per stride phase (dgrad with stride 2: four)
  int a_tma;
  int a_chunks;           // Cs / channels per chunk
  int stages;
  // k-blocks per stage (1 .. kMaxKps; more than one only with the A operand by TMA): the barriers of a
  // stage are passed once for all of its k-blocks, which halves the hand-offs between the producer, split
  // and MMA warps (each costs about a hundred nanoseconds whatever the work behind it)
  int kps;
  // fp32 (3xTF32) only: the K loop of a tile accumulates in nch chunks of kpc k-blocks, each in its own
  // BN TMEM columns (2 * BN with ts), summed by the epilogue; bf16 uses one chunk
  int kpc, nch;
  // fp32 with A by TMA: A in tensor memory. The producer warps split each landed A tile into tf32 hi / lo
  // and store both into a ring of TMEM stages (kTaKb k-blocks in all); per 8-wide k-step the MMAs run
  // D[:, 0:2BN] += A_hi x [B_hi; B_lo] and D[:, 0:BN] += A_lo x B_hi (B from shared memory, its lo rows
  // right after its hi rows), and the epilogue adds columns BN .. 2BN - 1 into 0 .. BN - 1. A shared-memory
  // stage then holds the raw A tile and B only, and the tensor core reads no A operand from shared memory
  int ts;
  // dgrad with every stride phase among the columns (phase-merged: the layer's phases all see the same
  // taps of the same d_conv neighbourhood): column c of row (n, a, b) is dX element (ph_h, r) =
  // (c / seg, c % seg) of the seg = S * IC contiguous values that start at pixel (S a + ph_h, S b), i.e.
  // phase column ph_w = r / IC, channel r % IC; seg_ld elements from one such run to the next row's; seg
  // and IC are powers of two, seg_sh and ic_sh their logarithms.
  // Runs of rows at or past out_h, and values of columns at or past out_w, are not written. 0: off.
  int seg, seg_sh, ic_sh, seg_ld, out_h, out_w;
  // bf16 dgrad of a 1x1, stride-1 batch-norm layer with d_conv formed in the A producer (no d_conv tensor):
  // a stage holds a k-block's pre-activation tile (tmap_a[0]) and dY tile (tmap_a[1]), 2-D boxes of 64
  // channels x 128 rows; warps 2-9 read them (half a row per thread), release the stage and write d_conv
  // into a ring of kTaKb TMEM stages (dconv_row_half), from which the MMAs take A; the same warps run the
  // epilogue one tile behind. B is resident (bres). xf_tbl: the per-channel terms [4][xf_C]. One k-block per
  // stage, single CTAs. 0: off.
  int xf, xf_C;
  const float* xf_tbl;
  // xf: the weights resident in shared memory behind the ring, bres bytes (one BN x 64 tile per k-block)
  uint32_t bres;
  // bf16 dgrad with d_conv by TMA: B read straight from the layer's weights W [OC][KH][KW][IC] as an MN-major
  // operand (no transposed copy): tmap_b is a 4-D view {64 input channels, OC, IC / 64 channel groups, KH * KW
  // taps}, and the k-block (tap counters tt, tw; output-channel chunk ck) of a phase takes the kernel tap
  // (rh + S (Th - 1 - tt), rw + S (Tw - 1 - tw)) (the flipped taps of the im2col order), oc ck * 64 ..: one copy
  // lands BN / 64 panels of 64 oc rows x 64 channels (128-byte swizzle). IC and BN multiples of 64. 0: off.
  int b_mn, S, KW;
  int* err;
  ConvPhase ph[kMaxPhases];
};

struct WgradParams {
  CUtensorMap tmap_dc;    // bf16 d_conv [n_pix][OCp], box {64 ch, 64 pix}
  CUtensorMap tmap_x;     // im2col map of X (when a_tma): bf16 64 pixels x 64 channels, fp32 32 x 32
  int a_tma;              // A by TMA im2col (Cs a multiple of 64 bf16 / 32 fp32). fp32: X and d_conv
                          // land as raw pixel-major tiles in a ring of rstages and the producer
                          // warps transpose them into tf32 hi / lo K-major stages
  int rstages;
  const void* x;          // NHWC [Nimg][H][W][Cs]
  const float* dc32;      // fp32 d_conv [n_pix][OCp] (fp32 mode)
  int H, W, Cs, OH, OW, S, P, KW;
  FastDiv div_Cs, div_KW, div_OW, div_OHOW;
  int Mk;                 // rows of D: KH*KW*Cs
  int m_tiles, n_tiles, BN, N, OCp;
  int n_pix, kb_total, kb_per_split, splits;
  int num_units;
  float* partial;         // [splits][N][Mk]
  int stages;
  int pair;               // CTA pairs (cta_group::2, bf16 with A by TMA): m_tiles counts pairs of m-tiles
  // bf16 with A by TMA: k-blocks per stage (1 or 2). With two, each copy covers both: the im2col panels and
  // the d_conv boxes are 64 * kps pixels tall, so a panel holds k-block i at 8 KB * i and the panels (and
  // the d_conv boxes) are kps * 8 KB apart; the barriers are passed once per two k-blocks
  int kps;
  // fp32 with raw TMA tiles: A (X, k rows x 32 pixels) in tensor memory, one TMEM stage per shared-memory
  // stage, which then holds the d_conv hi and lo rows only; the MMAs as in ConvGemmParams::ts
  int ts;
  // bf16 1x1, stride-1 layers: d_conv formed in the B producer (as ConvGemmParams::xf). A stage holds the X
  // panels (tmap_x), the pre-activation panels (tmap_dc) and the dY panels (tmap_dy), each brought by one
  // copy through a 3-D view of its [n_pix][channels] matrix (64 channels x pixels x 64-channel groups, boxes
  // of 64 x 64 x panels); warps 2-5 turn the pre-activation panels into d_conv. One k-block per stage,
  // single CTAs. 0: off.
  CUtensorMap tmap_dy;
  int xf, xf_C, act;      // act: the layer's activation (2 tanh or 3 sigmoid)
  const float* xf_tbl;
  int* err;
};

__host__ __device__ inline uint32_t tmem_cols_for(int cols) {
  uint32_t c = 32;
  while (c < static_cast<uint32_t>(cols)) c <<= 1;
  return c;
}

__device__ __forceinline__ const ConvPhase& find_phase(const ConvGemmParams& p, int u) {
  int i = 0;
  while (i + 1 < p.num_phases && p.ph[i + 1].unit_begin <= u) ++i;
  return p.ph[i];
}

// Value as stored in T (bf16: round to nearest even; fp32: unchanged).
template <typename T>
__device__ __forceinline__ float to_stored(float v);
template <>
__device__ __forceinline__ float to_stored<float>(float v) {
  return v;
}
template <>
__device__ __forceinline__ float to_stored<__nv_bfloat16>(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

// Column sums of a 32-row x 16-column block held one row per lane: a
// butterfly that halves the columns each lane keeps at every step. Afterwards
// 16 consecutive floats from shared memory (16-byte aligned) as four vector loads.
__device__ __forceinline__ void lds16(const float* p, float (&x)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 t = *reinterpret_cast<const float4*>(p + 4 * i);
    x[4 * i] = t.x;
    x[4 * i + 1] = t.y;
    x[4 * i + 2] = t.z;
    x[4 * i + 3] = t.w;
  }
}

// v = acc * scale + shift for 32 accumulator columns; scale and shift are per column in shared
// memory (16-byte aligned); without a scale only the shift is read.
__device__ __forceinline__ void ep_columns(const uint32_t (&r)[32], bool zero, bool has_scale, const float* sc,
                                           const float* sh, float (&v)[32]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float b[16];
    lds16(sh + 16 * h, b);
    if (zero) {  // no k-block reached the accumulator: v = shift (uniform branches below)
#pragma unroll
      for (int e = 0; e < 16; ++e) v[16 * h + e] = b[e];
    } else if (has_scale) {
      float a[16];
      lds16(sc + 16 * h, a);
#pragma unroll
      for (int e = 0; e < 16; e += 2) {
        const float2 x = __ffma2_rn(make_float2(__uint_as_float(r[16 * h + e]), __uint_as_float(r[16 * h + e + 1])),
                                    make_float2(a[e], a[e + 1]), make_float2(b[e], b[e + 1]));
        v[16 * h + e] = x.x;
        v[16 * h + e + 1] = x.y;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 16; e += 2) {
        const float2 x = __fadd2_rn(make_float2(__uint_as_float(r[16 * h + e]), __uint_as_float(r[16 * h + e + 1])),
                                    make_float2(b[e], b[e + 1]));
        v[16 * h + e] = x.x;
        v[16 * h + e + 1] = x.y;
      }
    }
  }
}

// One level of a transposed butterfly over lane bit O: the pairs (x[e], x[e + W/2]) are
// exchanged with lane L ^ O, lanes with bit O set keep (and add up) the upper half,
// the others the lower half; afterwards x[0 .. W/2) holds the kept sums.
template <int W, int O>
__device__ __forceinline__ void colsum_step(float (&x)[16], int lane) {
  const bool up = (lane & O) != 0;
#pragma unroll
  for (int e = 0; e < W / 2; ++e) {
    const float send = up ? x[e] : x[e + W / 2];
    const float keep = up ? x[e + W / 2] : x[e];
    x[e] = keep + __shfl_xor_sync(0xffffffffu, send, O);
  }
}

__device__ __forceinline__ float2 f2(uint32_t a, uint32_t b) { return make_float2(__uint_as_float(a), __uint_as_float(b)); }

// Column sums of d and of d*d over the 32 rows of this warp's TMEM lane quarter, for the 32
// accumulator columns at taddr, with d = acc * a + k per column (a = null: d = acc + k; k is
// the epilogue shift minus the statistics shift; both 8-byte aligned, indexed from the
// chunk's first column). Two 16-lane loads give thread t rows t/4 + {0, 8, 16, 24} of the
// column pairs 8j + 2(t%4) + {0, 1}: the four rows are added in the thread with packed
// f32x2 arithmetic, then a transposed butterfly over lane bits 4, 3, 2 leaves each lane one
// column pair of one statistic. rowmask bit i clears row t/4 + 8i (rows past the tile's
// end); zero: the accumulator was never written (read as 0). Writes sum(d) to s1[0..31]
// and sum(d*d) to s2[0..31]. Warp-collective. Kept out of line: inlined into both
// statistics passes it pushed the epilogue past the register budget of the 320-thread CTA.
static __device__ __noinline__ void colstats32(uint32_t taddr, bool zero, const float* a, const float* k, unsigned rowmask,
                                               int lane, float* s1, float* s2) {
  const int cp = 2 * (lane & 3);
  uint32_t r[2][16];
  if (zero) {
#pragma unroll
    for (int e = 0; e < 16; ++e) r[0][e] = r[1][e] = 0u;
  } else {  // both 16-lane halves in flight, one wait
    tmem_ld16x256(taddr, r[0]);
    tmem_ld16x256(taddr + (16u << 16), r[1]);
    tmem_ld_wait16x2(r[0], r[1]);
  }
  float x[16];  // x[2j + kk]: sum over the four rows of column 8j + cp + kk; x[8 + 2j + kk]: sum of squares
#pragma unroll
  for (int e = 0; e < 16; ++e) x[e] = 0.f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {  // lanes 0-15, then 16-31 of the quarter
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 kv = *reinterpret_cast<const float2*>(k + 8 * j + cp);
      float2 d0 = f2(r[h][4 * j], r[h][4 * j + 1]), d1 = f2(r[h][4 * j + 2], r[h][4 * j + 3]);
      if (a) {
        const float2 av = *reinterpret_cast<const float2*>(a + 8 * j + cp);
        d0 = __ffma2_rn(d0, av, kv);
        d1 = __ffma2_rn(d1, av, kv);
      } else {
        d0 = __fadd2_rn(d0, kv);
        d1 = __fadd2_rn(d1, kv);
      }
      if (rowmask != 0u) {
        if ((rowmask >> (2 * h)) & 1u) d0 = make_float2(0.f, 0.f);
        if ((rowmask >> (2 * h + 1)) & 1u) d1 = make_float2(0.f, 0.f);
      }
      float2 sv = make_float2(x[2 * j], x[2 * j + 1]), sq = make_float2(x[8 + 2 * j], x[8 + 2 * j + 1]);
      sv = __fadd2_rn(sv, __fadd2_rn(d0, d1));
      sq = __ffma2_rn(d0, d0, sq);
      sq = __ffma2_rn(d1, d1, sq);
      x[2 * j] = sv.x;
      x[2 * j + 1] = sv.y;
      x[8 + 2 * j] = sq.x;
      x[8 + 2 * j + 1] = sq.y;
    }
  }
  colsum_step<16, 16>(x, lane);  // lanes with bit 4 set keep the squares
  colsum_step<8, 8>(x, lane);    // bit 3: column groups j = 2, 3 (else 0, 1)
  colsum_step<4, 4>(x, lane);    // bit 2: the odd group of the two
  const int j = 2 * ((lane >> 3) & 1) + ((lane >> 2) & 1);
  float* dst = (lane & 16) ? s2 : s1;
  *reinterpret_cast<float2*>(dst + 8 * j + cp) = make_float2(x[0], x[1]);
}

// Sum the accumulator chunks 1 .. n-1 (n >= 2) of a tile into chunk 0, in fp32 round-to-nearest and
// chunk order: columns [c0, c1) (multiples of 32) of this warp's lane quarter, chunk i starting
// i * stride columns after taddr. The tensor core's fp32 accumulation loses a little on every MMA step;
// a deep K loop split over chunks keeps that loss to the steps of one chunk. With A in TMEM each chunk
// is itself two column blocks (see ConvGemmParams::ts). Warp-collective.
static __device__ __noinline__ void fold_chunks(uint32_t taddr, int stride, int n, int c0, int c1) {
  for (int c = c0; c < c1; c += 32) {
    uint32_t a[32], b[32];
    tmem_ld32(taddr + c, a);
    tmem_ld32(taddr + static_cast<uint32_t>(stride + c), b);
    tmem_ld_wait2(a, b);
#pragma unroll
    for (int e = 0; e < 32; ++e) a[e] = __float_as_uint(__uint_as_float(a[e]) + __uint_as_float(b[e]));
    for (int i = 2; i < n; ++i) {
      tmem_ld32(taddr + static_cast<uint32_t>(i * stride + c), b);
      tmem_ld_wait2(a, b);
#pragma unroll
      for (int e = 0; e < 32; ++e) a[e] = __float_as_uint(__uint_as_float(a[e]) + __uint_as_float(b[e]));
    }
    tmem_st32(taddr + c, a);
  }
  tmem_st_wait();
}

// d_conv of a batch-norm layer with training statistics from its stored pre-activation x and dY (bf16):
//   z = (x - mean) inv_std, t = gamma z + beta, d_norm = act'(t) dY,
//   d_conv = inv_std (gamma d_norm - k1 - z k2),  k1 = gamma sum(d_norm) / n,  k2 = gamma sum(d_norm z) / n,
// taken per channel as t = G x + B' and d_conv = G d_norm + Q x + S' (G = gamma inv_std, B' = beta - G mean,
// Q = -inv_std^2 k2, S' = -inv_std k1 - Q mean: bn_bwd_fused_finalize_kernel); bf16 layers take the fast
// activations, as the stand-alone d_conv pass does. Two channels: the packed bf16 pairs of x and dY in, the
// packed bf16 pair of d_conv out.
template <int A>
__device__ __forceinline__ uint32_t dconv_pair(uint32_t wx, uint32_t wd, float2 G, float2 Bp, float2 Q, float2 Sp) {
  const float2 x = make_float2(__uint_as_float(wx << 16), __uint_as_float(wx & 0xffff0000u));
  const float2 dy = make_float2(__uint_as_float(wd << 16), __uint_as_float(wd & 0xffff0000u));
  const float2 t = __ffma2_rn(G, x, Bp);
  float2 dn;
  if constexpr (A == 1) {
    dn = make_float2(t.x > 0.f ? dy.x : 0.f, t.y > 0.f ? dy.y : 0.f);
  } else {
    dn = make_float2(dact_t<A, true>(t.x) * dy.x, dact_t<A, true>(t.y) * dy.y);
  }
  const float2 v = __ffma2_rn(G, dn, __ffma2_rn(Q, x, Sp));
  __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
  return *reinterpret_cast<uint32_t*>(&h);
}

// d_conv formed in a shared-memory stage (see dconv_pair). The tiles are nbox boxes of NR * RS rows of 64
// channels (128-byte swizzle; box b at b * NR * RS * 128 bytes): x at xa, dY at the same offsets from ya;
// d_conv replaces x. Thread t (of 8 RS) takes 16-byte chunk t & 7 of rows t / 8 + RS i of every box; under
// the swizzle that chunk holds channels 8 ((t & 7) ^ (t / 8 & 7)) .. + 7 of the box in each of those rows.
// All NR rows of a box are read before any is computed. tbl: the terms [4][C] (G, B', Q, S') in shared
// memory; c0: channel of box 0's first column; channels at or past C take zero terms; rows at or past
// nvalid (pixels past the layer) are written as zeros.
template <int A, int NR, int RS>
__device__ __forceinline__ void dconv_xform(uint32_t xa, uint32_t ya, int nbox, const float* tbl, int C, int c0,
                                            int nvalid, int t) {
  const int pj = t & 7, r0 = t >> 3;
  const int ch = 8 * (pj ^ (r0 & 7));
  for (int b = 0; b < nbox; ++b) {
    const int c = c0 + 64 * b + ch;
    float k[4][8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
      if (c < C) {  // C is a multiple of 8: the thread's eight channels are all inside or all outside
        lo = *reinterpret_cast<const float4*>(tbl + q * C + c);
        hi = *reinterpret_cast<const float4*>(tbl + q * C + c + 4);
      }
      k[q][0] = lo.x; k[q][1] = lo.y; k[q][2] = lo.z; k[q][3] = lo.w;
      k[q][4] = hi.x; k[q][5] = hi.y; k[q][6] = hi.z; k[q][7] = hi.w;
    }
    const uint32_t bo = static_cast<uint32_t>(b * NR * RS * 128 + r0 * 128 + (pj << 4));
    uint32_t wx[NR][4], wd[NR][4];
#pragma unroll
    for (int i = 0; i < NR; ++i) {
      const uint32_t off = bo + static_cast<uint32_t>(i * RS * 128);
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(wx[i][0]), "=r"(wx[i][1]), "=r"(wx[i][2]), "=r"(wx[i][3]) : "r"(xa + off));
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(wd[i][0]), "=r"(wd[i][1]), "=r"(wd[i][2]), "=r"(wd[i][3]) : "r"(ya + off));
    }
#pragma unroll
    for (int i = 0; i < NR; ++i) {
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int e = 2 * q;
        const uint32_t v = dconv_pair<A>(wx[i][q], wd[i][q], make_float2(k[0][e], k[0][e + 1]),
                                         make_float2(k[1][e], k[1][e + 1]), make_float2(k[2][e], k[2][e + 1]),
                                         make_float2(k[3][e], k[3][e + 1]));
        o[q] = r0 + RS * i < nvalid ? v : 0u;
      }
      st_shared_v4(xa + bo + static_cast<uint32_t>(i * RS * 128), o[0], o[1], o[2], o[3]);
    }
  }
}

// d_conv of one half row of a 128-row x 64-channel stage (the calling thread's row r, its TMEM lane, and
// channels 32 H .. 32 H + 31) from the pre-activation tile at xa and the dY tile at ya (128-byte swizzle):
// dconv_row_load reads the half row's four 16-byte chunks of both (logical chunk cc at physical chunk
// cc ^ (r & 7)); dconv_row_half forms them as the 16 packed bf16 pairs of an A operand in tensor memory
// (column c = channels 2c, 2c + 1). tbl: the terms [4][C]; c0: channel of the tile's first column;
// zero = the row is past the layer (written as zeros).
__device__ __forceinline__ void dconv_row_load(uint32_t xa, uint32_t ya, int r, int H, uint32_t (&wx)[4][4],
                                               uint32_t (&wd)[4][4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int cc = 4 * H + i;
    const uint32_t off = static_cast<uint32_t>(r * 128 + ((cc ^ (r & 7)) << 4));
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(wx[i][0]), "=r"(wx[i][1]), "=r"(wx[i][2]), "=r"(wx[i][3]) : "r"(xa + off));
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(wd[i][0]), "=r"(wd[i][1]), "=r"(wd[i][2]), "=r"(wd[i][3]) : "r"(ya + off));
  }
}
template <int A>
__device__ __forceinline__ void dconv_row_half(const uint32_t (&wx)[4][4], const uint32_t (&wd)[4][4], int H,
                                               const float* tbl, int C, int c0, bool zero, uint32_t (&o)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float* k = tbl + c0 + 8 * (4 * H + i);  // the same channels in every lane: broadcast reads
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float4 g = *reinterpret_cast<const float4*>(k + 4 * h);
      const float4 bp = *reinterpret_cast<const float4*>(k + C + 4 * h);
      const float4 qq = *reinterpret_cast<const float4*>(k + 2 * C + 4 * h);
      const float4 sp = *reinterpret_cast<const float4*>(k + 3 * C + 4 * h);
      const uint32_t v0 = dconv_pair<A>(wx[i][2 * h], wd[i][2 * h], make_float2(g.x, g.y), make_float2(bp.x, bp.y),
                                        make_float2(qq.x, qq.y), make_float2(sp.x, sp.y));
      const uint32_t v1 = dconv_pair<A>(wx[i][2 * h + 1], wd[i][2 * h + 1], make_float2(g.z, g.w),
                                        make_float2(bp.z, bp.w), make_float2(qq.z, qq.w), make_float2(sp.z, sp.w));
      o[4 * i + 2 * h] = zero ? 0u : v0;
      o[4 * i + 2 * h + 1] = zero ? 0u : v1;
    }
  }
}

// The per-channel terms of d_conv [4][C] (C a multiple of 8) copied into shared memory by the nthr threads
// of the transforming warps, which then pass named barrier 2 together.
__device__ __forceinline__ void load_xform_terms(float* dst, const float* __restrict__ src, int C, int t, int nthr) {
  for (int i = 4 * t; i < 4 * C; i += 4 * nthr)
    *reinterpret_cast<float4*>(dst + i) = __ldg(reinterpret_cast<const float4*>(src + i));
  named_bar_sync(2, nthr);
}

template <typename T>
__device__ __forceinline__ void store_row16(T* dst, const float* v, int ncols, bool vec);

template <>
__device__ __forceinline__ void store_row16<__nv_bfloat16>(__nv_bfloat16* dst, const float* v, int ncols, bool vec) {
  if (vec && ncols >= 16) {
    uint32_t w[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
      w[e] = *reinterpret_cast<uint32_t*>(&h);
    }
    reinterpret_cast<uint4*>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
    reinterpret_cast<uint4*>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
  } else {
#pragma unroll
    for (int e = 0; e < 16; ++e)
      if (e < ncols) dst[e] = __float2bfloat16_rn(v[e]);
  }
}
template <>
__device__ __forceinline__ void store_row16<float>(float* dst, const float* v, int ncols, bool vec) {
  if (vec && ncols >= 16) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      reinterpret_cast<float4*>(dst)[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
  } else {
#pragma unroll
    for (int e = 0; e < 16; ++e)
      if (e < ncols) dst[e] = v[e];
  }
}

// 32 columns col0 .. col0 + 31 of a phase-merged dgrad row (ConvGemmParams::seg) whose first output pixel
// (h0, w0) = (S a, S b) is at out + obase. seg = S * IC divides 32, so it and IC are powers of two (seg_sh,
// ic_sh their logarithms) and every 16-byte group of columns lies inside one run of seg contiguous dX
// values; the groups are unrolled so that v stays in registers.
template <typename T>
__device__ __forceinline__ void store_phase_runs(T* out, size_t obase, int h0, int w0, int col0, const float (&v)[32],
                                                 int ncols, const ConvGemmParams& p) {
  constexpr int EC = 16 / sizeof(T);
  const bool whole = w0 + (p.seg >> p.ic_sh) <= p.out_w;  // every phase column of a run inside the image
#pragma unroll
  for (int e = 0; e < 32; e += EC) {
    if (e < ncols) {
      const int c = col0 + e;
      const int ph_h = c >> p.seg_sh, r = c - (ph_h << p.seg_sh);
      if (h0 + ph_h < p.out_h) {
        T* dst = out + obase + static_cast<size_t>(ph_h) * p.seg_ld + r;
        if (whole) {
          if constexpr (sizeof(T) == 4) {
            *reinterpret_cast<float4*>(dst) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
          } else {
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              __nv_bfloat162 h = __floats2bfloat162_rn(v[e + 2 * q], v[e + 2 * q + 1]);
              w[q] = *reinterpret_cast<uint32_t*>(&h);
            }
            *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
#pragma unroll
          for (int q = 0; q < EC; ++q)
            if (w0 + ((r + q) >> p.ic_sh) < p.out_w) dst[q] = static_cast<T>(v[e + q]);
        }
      }
    }
  }
}

// 32 bytes to global memory in one store (the address 32-byte aligned): a whole sector per lane
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t* w) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// 32 values of a row to T at dst: 16-byte stores (vec: dst 16-byte aligned), for bf16 32-byte ones (vec32:
// dst 32-byte aligned), else one value at a time; columns at or past ncols are not written.
template <typename T>
__device__ __forceinline__ void store_row32(T* dst, const float (&v)[32], int ncols, bool vec, bool vec32 = false) {
  if (vec && ncols >= 32) {
    if constexpr (sizeof(T) == 2) {
      uint32_t w[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
        w[e] = *reinterpret_cast<uint32_t*>(&h);
      }
      if (vec32) {
        st_global_v8(dst, w);
        st_global_v8(dst + 16, w + 8);
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          reinterpret_cast<uint4*>(dst)[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        reinterpret_cast<float4*>(dst)[e] = make_float4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 32; ++e)
      if (e < ncols) dst[e] = static_cast<T>(v[e]);
  }
}

// --------------------------------------------------------------------------
// fprop / dgrad
// --------------------------------------------------------------------------
// PAIR: CTA pairs (cta_group::2); bf16 with A by TMA and one phase only. A kernel may not mix
// single-CTA and pair tcgen05 forms, hence the separate instantiation. BMN: B read straight from the
// weights as an MN-major operand (ConvGemmParams::b_mn), an instantiation of its own so that the other
// GEMMs' MMA loop carries no test of it.
template <int DT, bool PAIR, bool BMN = false>
__global__ void __launch_bounds__(kThreads, 1) conv_gemm_kernel(const __grid_constant__ ConvGemmParams p) {
  pdl_entry();
  using D = Dt<DT>;
  using T = typename D::T;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int BN = p.BN;
  constexpr bool pair = PAIR;
  static_assert(!PAIR || DT == 1, "CTA pairs run bf16 only");
  static_assert(!BMN || DT == 1, "weights read as an MN-major operand in bf16 only");
  const uint32_t a_bytes = kBM * 128, b_bytes = BN * 128;
  // a pair member holds its 128 rows of A and half of B's columns
  const uint32_t b_own = pair ? b_bytes / 2 : b_bytes;
  // fp32 with A in TMEM (see ConvGemmParams::ts): a stage holds the raw A tile, B hi and B lo
  const bool ts = DT == 0 && p.ts;
  // d_conv formed from the pre-activation and dY tiles into tensor memory (see ConvGemmParams::xf): a
  // stage holds those two tiles only, and B is resident behind the ring
  const bool xf = DT == 1 && !PAIR && p.xf;
  const uint32_t a_tiles = (DT == 0 && !ts) ? 2u : 1u;  // A tiles per k-block (fp32 in shared memory: hi, lo)
  const int KPS = p.kps > 1 ? p.kps : 1;                // k-blocks per stage
  const uint32_t sub_bytes = xf ? 2 * a_bytes : a_tiles * a_bytes + D::NS * b_own;  // one k-block of a stage
  const uint32_t stage_bytes = KPS * sub_bytes;
  const int S = p.stages;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * stage_bytes + (xf ? p.bres : 0u));
  uint64_t* empty = full + kMaxStages;
  uint64_t* tfull = empty + kMaxStages;
  uint64_t* tempty = tfull + kMaxTmemBufs;
  uint64_t* sfull = tempty + kMaxTmemBufs;  // fp32 with A by TMA: the stage is split into hi / lo
  uint64_t* aempty = sfull + kMaxStages;    // A in TMEM: the MMAs have read a TMEM stage of A
  uint64_t* bfull = &sfull[kMaxStages - 1];  // xf: the resident B tiles have landed (TA < kMaxStages - 1)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(aempty + kMaxStages);
  const uint32_t sbase = smem_u32(smem);
  // fp32 with A by TMA: warps 2-5 split the stages (and the epilogue keeps four warps)
  const bool split_a = DT == 0 && p.a_tma;
  // epilogue of eight warps (warps 2-9) when the gather warps are free: bf16 with A by TMA
  const bool ep8 = DT == 1 && p.a_tma && !xf;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = pair ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;  // issues the MMAs of the pair
  // units this CTA (pair) walks: pairs of m-tiles when paired
  const int cid = pair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int ncl = pair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  // TMEM accumulators in flight: as many BN-column buffers as fit (at least two), so that short tiles
  // (few k-blocks) keep the MMA busy while the epilogue of earlier tiles completes
  // fp32: nch accumulator chunks of BN columns per tile (see ConvGemmParams::kpc)
  const int nch = DT == 0 && p.nch > 1 ? p.nch : 1;
  const int kpc = DT == 0 && p.nch > 1 ? p.kpc : (1 << 30);
  const int ccols = ts ? 2 * BN : BN;  // TMEM columns of one accumulator chunk
  const int tcs = nch * ccols;         // TMEM columns of one tile
  // with A in TMEM the last columns hold TA stages of KPS k-blocks of A (fp32: per k-block hi, 32 columns,
  // then lo, 32; xf: 32 columns of packed bf16 pairs per k-block)
  const int TA = kTaKb / KPS;
  const int ta_cols = ts ? kTaKb * 64 : (xf ? kTaKb * 32 : 0);
  const int nbuf = (512 - ta_cols) / tcs < kMaxTmemBufs ? (512 - ta_cols) / tcs : kMaxTmemBufs;
  const uint32_t tcols = tmem_cols_for(nbuf * tcs + ta_cols);
  const uint32_t ta0 = static_cast<uint32_t>(nbuf * tcs);  // first TMEM column of the A stages

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], p.a_tma ? 1 : 4 + 1);  // the TMA thread (+ one arrival per producer warp)
      mbar_init(&empty[s], xf ? 8 : 1);          // the MMA's commit (xf: one arrival per transforming warp)
    }
    for (int b = 0; b < nbuf; ++b) {
      mbar_init(&tfull[b], 1);
      // one arrival per epilogue warp (of both CTAs when paired: the even CTA's MMA writes both TMEMs)
      mbar_init(&tempty[b], ((ep8 || xf) ? 8 : 4) * (pair ? 2 : 1));
    }
    if (split_a || xf)  // with A in TMEM indexed by TMEM stage; one arrival per splitting / transforming warp
      for (int s = 0; s < ((ts || xf) ? TA : S); ++s) mbar_init(&sfull[s], xf ? 8 : 4);
    if (ts || xf)
      for (int j = 0; j < TA; ++j) mbar_init(&aempty[j], 1);  // the MMA warp's commit
    if (xf) mbar_init(bfull, 1);
    fence_mbar_init();
    tma_prefetch_desc(&p.tmap_b);
    if (p.a_tma)
      for (int i = 0; i < p.num_phases && i < kMaxTmaPhases; ++i) tma_prefetch_desc(&p.tmap_a[i]);
    if (xf) tma_prefetch_desc(&p.tmap_a[1]);
  }
  if (warp == 1) {
    if (pair) {
      tmem_alloc_pair(tmem_slot, tcols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, tcols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (pair) cluster_sync();  // the peer's barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------ B producer (TMA)
    if (lane == 0 && xf) {
      // the resident B tiles once (one column tile), then the pre-activation and dY tiles of every k-block
      const uint32_t bres = sbase + S * stage_bytes;  // the resident B tiles, one per k-block
      const ConvPhase& ph0 = p.ph[0];
      mbar_arrive_expect_tx(bfull, p.bres);
      for (int kb = 0; kb < ph0.num_kb; ++kb) tma_load_2d(bres + kb * b_bytes, &p.tmap_b, bfull, ph0.b_col + kb * D::BKE, 0);
      int s = 0;
      uint32_t par = 0;
      bool alive = true;
      for (int u = cid; u < p.num_units && alive; u += ncl) {
        const ConvPhase& ph = find_phase(p, u);
        const int row0 = ((u - ph.unit_begin) / p.n_tiles) * kBM;
        for (int kb = 0; kb < ph.num_kb; ++kb) {
          if (!wait(&empty[s], par ^ 1, p.err, kSiteEmpty)) {
            alive = false;
            break;
          }
          const uint32_t a0 = sbase + s * stage_bytes;
          mbar_arrive_expect_tx(&full[s], 2 * a_bytes);
          tma_load_2d(a0, &p.tmap_a[0], &full[s], kb * D::BKE, row0);
          tma_load_2d(a0 + a_bytes, &p.tmap_a[1], &full[s], kb * D::BKE, row0);
          if (++s == S) {
            s = 0;
            par ^= 1;
          }
        }
      }
    } else if (lane == 0) {
      int s = 0;
      uint32_t par = 0;
      bool alive = true;
      for (int u = cid; u < p.num_units && alive; u += ncl) {
        const ConvPhase& ph = find_phase(p, u);
        const int local = u - ph.unit_begin;
        const int n_tile = local % p.n_tiles;
        int an = 0, ah = 0, aw = 0;  // window corner of the tile's first row (TMA im2col)
        if (p.a_tma) {
          const int m_tile = pair ? 2 * (local / p.n_tiles) + static_cast<int>(rank) : local / p.n_tiles;
          const int m0 = m_tile * kBM;
          an = static_cast<int>(fdiv(static_cast<uint32_t>(m0), ph.div_HaWa));
          const int rem = m0 - an * ph.Ha * ph.Wa;
          const int a = static_cast<int>(fdiv(static_cast<uint32_t>(rem), ph.div_Wa));
          ah = a * p.rs + ph.a_lo_h;
          aw = (rem - a * ph.Wa) * p.rs + ph.a_lo_w;
        }
        // im2col offsets of k-block kb = (tt * Tw + tw) * a_chunks + ck, advanced by counters (this thread
        // issues every copy of the CTA, so its per-k-block path is kept free of divisions)
        int ck = 0, tw = 0, tt = 0;
        for (int g0 = 0; g0 < ph.num_kb; g0 += KPS) {  // one stage: k-blocks g0 .. g0 + nk - 1
          const int nk = min(KPS, ph.num_kb - g0);
          if (!wait(&empty[s], par ^ 1, p.err, kSiteEmpty)) {
            alive = false;
            break;
          }
          // both pair members' loads complete on the even CTA's full barrier, which expects them all
          const uint32_t bar = pair ? mapa_shared(smem_u32(&full[s]), 0) : 0u;
          if (pair) {
            if (leader) mbar_arrive_expect_tx(&full[s], 2u * nk * (a_bytes + b_own));
          } else {
            mbar_arrive_expect_tx(&full[s], nk * (D::NS * b_bytes + (p.a_tma ? a_bytes : 0u)));
          }
#pragma unroll
          for (int i = 0; i < kMaxKps; ++i) {
            if (i >= nk) break;
            const int kcol = ph.b_col + (g0 + i) * D::BKE;
            const uint32_t a0 = sbase + s * stage_bytes + i * sub_bytes;
            const uint32_t b0 = a0 + a_tiles * a_bytes;
            // BMN: the kernel tap of this k-block (the flipped im2col order)
            const int wtap = BMN ? (ph.rh + p.S * (ph.Th - 1 - tt)) * p.KW + ph.rw + p.S * (ph.Tw - 1 - tw) : 0;
            if (pair) {
              tma_load_im2col_4d_pair(a0, &p.tmap_a[ph.a_map], bar, ck * D::BKE, aw, ah, an, static_cast<uint16_t>(tw),
                                      static_cast<uint16_t>(tt));
              if (BMN)
                tma_load_4d_pair(b0, &p.tmap_b, bar, 0, ck * D::BKE, (n_tile * BN + static_cast<int>(rank) * (BN / 2)) / 64,
                                 wtap);
              else
                tma_load_2d_pair(b0, &p.tmap_b, bar, kcol, n_tile * BN + static_cast<int>(rank) * (BN / 2));
            } else if (BMN) {
              tma_load_im2col_4d(a0, &p.tmap_a[ph.a_map], &full[s], ck * D::BKE, aw, ah, an, static_cast<uint16_t>(tw),
                                 static_cast<uint16_t>(tt));
              tma_load_4d(b0, &p.tmap_b, &full[s], 0, ck * D::BKE, n_tile * BN / 64, wtap);
            } else {
              if (p.a_tma)
                tma_load_im2col_4d(a0, &p.tmap_a[ph.a_map], &full[s], ck * D::BKE, aw, ah, an,
                                   static_cast<uint16_t>(tw), static_cast<uint16_t>(tt));
              if (D::NS == 2) tma_load_3d(b0, &p.tmap_b, &full[s], kcol, n_tile * BN, 0);  // hi and lo rows
              else tma_load_2d(b0, &p.tmap_b, &full[s], kcol, n_tile * BN);
            }
            if (++ck == p.a_chunks) {  // (without A by TMA a_chunks is 0 and the counters are unused)
              ck = 0;
              if (++tw == ph.Tw) {
                tw = 0;
                ++tt;
              }
            }
          }
          if (++s == S) {
            s = 0;
            par ^= 1;
          }
        }
      }
      if (pair) {
        // the even CTA's commits land in this CTA's empty barriers: let every stage's last use finish
        // before the CTA can exit
        for (int i = 0; i < S && alive; ++i) {
          if (!wait(&empty[s], par ^ 1, p.err, kSiteEmpty)) break;
          if (++s == S) {
            s = 0;
            par ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0 && xf) {
      // A (d_conv) from the TMEM stages the transforming warps fill, B from the resident tiles
      const uint32_t bres = sbase + S * stage_bytes;
      const uint32_t idesc = idesc_f32acc(kBM, BN, D::FMT, false, false);
      int j = 0, tc = 0;
      uint32_t apar = 0;
      bool alive = wait(bfull, 0, p.err, kSiteFull);
      for (int u = cid; u < p.num_units && alive; u += ncl, ++tc) {
        const ConvPhase& ph = find_phase(p, u);
        const int buf = tc % nbuf;
        if (!wait(&tempty[buf], ((tc / nbuf) & 1) ^ 1, p.err, kSiteTEmpty)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * tcs;
        for (int kb = 0; kb < ph.num_kb; ++kb) {
          if (!wait(&sfull[j], apar, p.err, kSiteFull)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = tmem_base + ta0 + static_cast<uint32_t>(j * 32);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ta(d, a + kk * 8, sdesc_sw128(bres + kb * b_bytes + kk * 32, 16, 1024), idesc, (kb | kk) ? 1u : 0u);
          mma_commit(&aempty[j]);
          if (++j == TA) {
            j = 0;
            apar ^= 1;
          }
        }
        if (alive) mma_commit(&tfull[buf]);
      }
    } else if (lane == 0 && leader) {
      const uint32_t idesc = idesc_f32acc(pair ? 2 * kBM : kBM, BN, D::FMT, false, BMN);
      const uint32_t idesc2 = idesc_f32acc(kBM, 2 * BN, D::FMT, false, false);  // A_hi x [B_hi; B_lo]
      int s = 0, j = 0;
      uint32_t par = 0, apar = 0;
      int tc = 0;
      bool alive = true;
      for (int u = cid; u < p.num_units && alive; u += ncl, ++tc) {
        const ConvPhase& ph = find_phase(p, u);
        const int buf = tc % nbuf;
        if (!wait(&tempty[buf], ((tc / nbuf) & 1) ^ 1, p.err, kSiteTEmpty)) break;
        tc_fence_after();
        const uint32_t dt = tmem_base + buf * tcs;
        for (int g0 = 0; g0 < ph.num_kb; g0 += KPS) {  // one stage: k-blocks g0 .. g0 + nk - 1
          const int nk = min(KPS, ph.num_kb - g0);
          // with A in TMEM the split warps arrive on the TMEM stage's barrier after the shared-memory stage
          // has landed, so that one wait covers both
          if (!wait(ts ? &sfull[j] : (split_a ? &sfull[s] : &full[s]), ts ? apar : par, p.err, kSiteFull)) {
            alive = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int i = 0; i < kMaxKps; ++i) {
            if (i >= nk) break;
            const int kb = g0 + i;
            const uint32_t d = DT == 0 ? dt + static_cast<uint32_t>((kb / kpc) * ccols) : dt;
            const int kc = DT == 0 ? kb % kpc : kb;  // k-block within the accumulator chunk
            const uint32_t a0 = sbase + s * stage_bytes + i * sub_bytes;
            const uint32_t b0 = a0 + a_tiles * a_bytes;
            if (ts) {
              const uint32_t ah = tmem_base + ta0 + static_cast<uint32_t>((j * KPS + i) * 64), al = ah + 32;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bd = sdesc_sw128(b0 + kk * 32, 16, 1024);  // 2 BN rows: hi, then lo
                mma_tf32_ta(d, ah + kk * 8, bd, idesc2, (kc | kk) ? 1u : 0u);
                mma_tf32_ta(d, al + kk * 8, bd, idesc, 1u);
              }
              continue;
            }
#pragma unroll
            for (int kk = 0; kk < 128 / 32; ++kk) {
              const uint64_t ad = sdesc_sw128(a0 + kk * 32, 16, 1024);
              // BMN: 16 oc rows (2 KB) of every 8 KB panel per k-step
              const uint64_t bd = BMN ? sdesc_sw128(b0 + kk * 2048, 8192, 1024) : sdesc_sw128(b0 + kk * 32, 16, 1024);
              const uint32_t acc = (kc | kk) ? 1u : 0u;
              if (DT == 1) {
                if (pair) mma_bf16_pair(d, ad, bd, idesc, acc);
                else mma_bf16(d, ad, bd, idesc, acc);
              } else {
                const uint64_t al = sdesc_sw128(a0 + a_bytes + kk * 32, 16, 1024);
                const uint64_t bl = sdesc_sw128(b0 + b_bytes + kk * 32, 16, 1024);
                mma_tf32(d, al, bd, idesc, acc);
                mma_tf32(d, ad, bl, idesc, 1u);
                mma_tf32(d, ad, bd, idesc, 1u);
              }
            }
          }
          if (pair) mma_commit_pair(&empty[s]);
          else mma_commit(&empty[s]);
          if (ts) mma_commit(&aempty[j]);
          if (++s == S) {
            s = 0;
            par ^= 1;
          }
          if (ts && ++j == TA) {
            j = 0;
            apar ^= 1;
          }
        }
        if (alive) {
          if (pair) mma_commit_pair(&tfull[buf]);
          else mma_commit(&tfull[buf]);
        }
      }
    }
  } else if (warp < 6 && !p.a_tma) {
    // ------------------------------------------------ A producers (gather)
    // (when the A operand comes by TMA im2col these warps join the epilogue)
    const int t = threadIdx.x - 64;
    const int j = t & 7;       // 16-byte chunk within the 128-byte row
    const int r0 = t >> 3;     // rows r0 + 16*i
    const uint32_t swz = static_cast<uint32_t>((j ^ (r0 & 7)) << 4);
    const char* src = static_cast<const char*>(p.src);
    int s = 0;
    uint32_t par = 0;
    int it = 0;
    bool alive = !p.a_tma;
    // k-blocks whose copies stay in flight before the stage is released (fewer when the ring is short).
    // fp32 keeps one: its stages are twice as large (hi and lo tiles), so the ring holds only 3-5 of
    // them, and every k-block of lag is a stage the MMA cannot use as slack.
    const int lag = DT == 0 ? 1 : (S - 1 < kLag ? S - 1 : kLag);
    // fp32: the copied rows land in the hi tile; once they are in, each thread splits its own chunks in
    // place (hi stays, lo goes to the lo tile)
    auto split_stage = [&](int q) {
      const uint32_t b0 = sbase + (q % S) * stage_bytes;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t dst = b0 + (r0 + 16 * i) * 128 + swz;
        uint32_t x0, x1, x2, x3;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3) : "r"(dst));
        uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
        split_tf32x2(__uint_as_float(x0), __uint_as_float(x1), h0, l0, h1, l1);
        split_tf32x2(__uint_as_float(x2), __uint_as_float(x3), h2, l2, h3, l3);
        st_shared_v4(dst, h0, h1, h2, h3);
        st_shared_v4(dst + a_bytes, l0, l1, l2, l3);
      }
    };
    // wait for all but the newest `lag` copy groups (an immediate operand, hence the switch)
    auto wait_lag = [&]() {
      if (lag >= 3) cp_async_wait<3>();
      else if (lag == 2) cp_async_wait<2>();
      else if (lag == 1) cp_async_wait<1>();
      else cp_async_wait<0>();
    };
    for (int u = blockIdx.x; u < p.num_units && alive; u += gridDim.x) {
      const ConvPhase& ph = find_phase(p, u);
      const int m_tile = (u - ph.unit_begin) / p.n_tiles;
      int hb[8], wb[8], pb[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int m = m_tile * kBM + r0 + 16 * i;
        if (m < ph.rows) {
          const int n = static_cast<int>(fdiv(static_cast<uint32_t>(m), ph.div_HaWa));
          const int rem = m - n * ph.Ha * ph.Wa;
          const int a = static_cast<int>(fdiv(static_cast<uint32_t>(rem), ph.div_Wa));
          const int b = rem - a * ph.Wa;
          hb[i] = a * p.rs + ph.qh;
          wb[i] = b * p.rs + ph.qw;
          pb[i] = n * p.Hs * p.Ws;
        } else {
          hb[i] = -(1 << 28);  // never in bounds
          wb[i] = 0;
          pb[i] = 0;
        }
      }
      for (int kb = 0; kb < ph.num_kb; ++kb) {
        const int k0 = kb * D::BKE + j * D::EC;
        const bool okc = k0 < ph.K;
        const int tap = static_cast<int>(fdiv(static_cast<uint32_t>(k0), p.div_Cs));
        const int c = k0 - tap * p.Cs;
        const int tt = static_cast<int>(fdiv(static_cast<uint32_t>(tap), ph.div_Tw));
        const int dh = p.tap_sign * tt;
        const int dw = p.tap_sign * (tap - tt * ph.Tw);
        if (!__all_sync(0xffffffffu, wait(&empty[s], par ^ 1, p.err, kSiteEmpty))) {  // warp-uniform
          alive = false;
          break;
        }
        const uint32_t a0 = sbase + s * stage_bytes;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int ih = hb[i] + dh, iw = wb[i] + dw;
          const bool ok = okc && static_cast<unsigned>(ih) < static_cast<unsigned>(p.Hs) &&
                          static_cast<unsigned>(iw) < static_cast<unsigned>(p.Ws);
          const size_t off = ok ? (static_cast<size_t>(pb[i] + ih * p.Ws + iw) * p.Cs + c) * D::ES : 0;
          const uint32_t dst = a0 + (r0 + 16 * i) * 128 + swz;
          cp_async16(dst, src + off, ok ? 16u : 0u);  // out of bounds: 16 zero bytes
        }
        cp_async_commit();
        if (it >= lag) {
          wait_lag();
          if (DT == 0) split_stage(it - lag);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&full[(it - lag) % S]);
        }
        ++it;
        if (++s == S) {
          s = 0;
          par ^= 1;
        }
      }
    }
    // the last `lag` stages: wait for every copy, split, release
    cp_async_wait<0>();
    if (alive) {
      for (int q = (it > lag ? it - lag : 0); q < it; ++q) {
        if (DT == 0) split_stage(q);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[q % S]);
      }
    }
  } else if (warp < 6 && ts) {
    // ------------------------------------------------ fp32 A split into TMEM (A by TMA)
    // Warp w owns TMEM lane quarter w & 3, i.e. rows 32 (w & 3) .. + 31 of the A tiles; for each k-block
    // of the landed stage each thread reads its row (32 channels, eight 16-byte chunks of the 128-byte
    // swizzle), splits it into tf32 hi / lo and stores both into its 64 columns of TMEM stage j (hi:
    // columns 0-31, lo: 32-63; column = k).
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ta0;
    int s = 0, j = 0;
    uint32_t par = 0, apar = 0;
    bool alive = true;
    for (int u = cid; u < p.num_units && alive; u += ncl) {
      const ConvPhase& ph = find_phase(p, u);
      for (int g0 = 0; g0 < ph.num_kb; g0 += KPS) {  // one stage: k-blocks g0 .. g0 + nk - 1
        const int nk = min(KPS, ph.num_kb - g0);
        // the raw tiles have landed, and the MMAs that read TMEM stage j before have completed
        const bool ok = wait(&full[s], par, p.err, kSiteFull) && wait(&aempty[j], apar ^ 1, p.err, kSiteEmpty);
        if (!__all_sync(0xffffffffu, ok)) {  // warp-uniform
          alive = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int i = 0; i < kMaxKps; ++i) {
          if (i >= nk) break;
          const uint32_t src = sbase + s * stage_bytes + i * sub_bytes + r * 128;
          const uint32_t dst = tq + static_cast<uint32_t>((j * KPS + i) * 64);
#pragma unroll
          for (int h = 0; h < 2; ++h) {  // channels 16h .. 16h + 15
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int cc = 4 * h + c;
              uint32_t x0, x1, x2, x3;
              asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                           : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                           : "r"(src + ((cc ^ (r & 7)) << 4)));
              split_tf32x2(__uint_as_float(x0), __uint_as_float(x1), hi[4 * c], lo[4 * c], hi[4 * c + 1],
                           lo[4 * c + 1]);
              split_tf32x2(__uint_as_float(x2), __uint_as_float(x3), hi[4 * c + 2], lo[4 * c + 2], hi[4 * c + 3],
                           lo[4 * c + 3]);
            }
            tmem_st16(dst + 16 * h, hi);
            tmem_st16(dst + 32 + 16 * h, lo);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfull[j]);
        if (++s == S) {
          s = 0;
          par ^= 1;
        }
        if (++j == TA) {
          j = 0;
          apar ^= 1;
        }
      }
    }
  } else if (warp < 6 && split_a) {
    // ------------------------------------------------ fp32 stage split (A by TMA)
    // each thread splits its eight 16-byte chunks of the stage's A tile in place: hi stays, lo goes
    // to the lo tile (the chunk layout of the TMA's 128-byte swizzle does not matter to an
    // element-wise split)
    const int t = threadIdx.x - 64;
    const int j = t & 7, r0 = t >> 3;
    const uint32_t swz = static_cast<uint32_t>((j ^ (r0 & 7)) << 4);
    int s = 0;
    uint32_t par = 0;
    bool alive = true;
    for (int u = cid; u < p.num_units && alive; u += ncl) {
      const ConvPhase& ph = find_phase(p, u);
      for (int kb = 0; kb < ph.num_kb; ++kb) {
        if (!__all_sync(0xffffffffu, wait(&full[s], par, p.err, kSiteFull))) {  // warp-uniform
          alive = false;
          break;
        }
        const uint32_t a0 = sbase + s * stage_bytes;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint32_t dst = a0 + (r0 + 16 * i) * 128 + swz;
          uint32_t x0, x1, x2, x3;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3) : "r"(dst));
          uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
          split_tf32x2(__uint_as_float(x0), __uint_as_float(x1), h0, l0, h1, l1);
          split_tf32x2(__uint_as_float(x2), __uint_as_float(x3), h2, l2, h3, l3);
          st_shared_v4(dst, h0, h1, h2, h3);
          st_shared_v4(dst + a_bytes, l0, l1, l2, l3);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfull[s]);
        if (++s == S) {
          s = 0;
          par ^= 1;
        }
      }
    }
  } else if (xf) {
    // ------------------------------------------------ d_conv into TMEM, and the epilogue
    // Warps w and w + 4 (w = 2..5) own TMEM lane quarter w & 3, i.e. rows 32 (w & 3) .. + 31 of a tile, and
    // channel half h = (w - 2) / 4 of each k-block: each thread reads its half row of both tiles, releases
    // the stage to the producer, and writes 16 columns of packed bf16 pairs of d_conv into TMEM stage j once
    // the MMAs of its previous use have completed. After a tile's k-blocks the eight warps store the tile
    // before it (its accumulator completed meanwhile), each its lane quarter and column half. The terms of
    // d_conv follow the epilogue scratch.
    const int q = warp & 3, h = (warp - 2) >> 2;
    const int r = q * 32 + lane;
    float* tbl = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(tmem_slot) + 16) + 12 * BN;
    load_xform_terms(tbl, p.xf_tbl, p.xf_C, threadIdx.x - 64, 256);
    const uint32_t tq = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ta0 + 16 * h;
    const int hcols = 32 * ((BN / 32 + 1) / 2);
    const int cb = h * hcols, ce = h ? BN : hcols;
    const bool vec = (p.out_ld % D::EC) == 0;
    const bool vec32 = vec && (((static_cast<size_t>(p.out_ld) * sizeof(T)) | reinterpret_cast<uintptr_t>(p.out)) & 31u) == 0;
    // store tile u (the tc-th of this CTA): a 1x1, stride-1 dgrad writes row m of D to dX pixel m
    auto epilogue = [&](int u, int tc) -> bool {
      const ConvPhase& ph = find_phase(p, u);
      const int local = u - ph.unit_begin;
      const int m_tile = local / p.n_tiles, n_tile = local % p.n_tiles;
      const int buf = tc % nbuf;
      int ok = 1;
      if (lane == 0) ok = wait(&tfull[buf], (tc / nbuf) & 1, p.err, kSiteTFull) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
      tc_fence_after();
      const int m = m_tile * kBM + r;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * tcs;
      T* out = static_cast<T*>(p.out) + static_cast<size_t>(m) * p.out_ld;
      for (int c0 = cb; c0 < ce; c0 += 64) {  // 64 columns per wait (two 32-column loads)
        if (n_tile * BN + c0 >= p.N) break;  // uniform across the warp
        const int c1 = c0 + 32 < ce ? c0 + 32 : c0;
        uint32_t ra[32], rb[32];
        tmem_ld32(taddr + c0, ra);
        tmem_ld32(taddr + c1, rb);
        tmem_ld_wait2(ra, rb);
        float v[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(ra[e]);
        if (m < ph.rows) store_row32<T>(out + n_tile * BN + c0, v, p.N - (n_tile * BN + c0), vec, vec32);
        if (c1 != c0 && n_tile * BN + c1 < p.N) {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(rb[e]);
          if (m < ph.rows) store_row32<T>(out + n_tile * BN + c1, v, p.N - (n_tile * BN + c1), vec, vec32);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
      return true;
    };
    int s = 0, j = 0;
    uint32_t par = 0, apar = 0;
    bool alive = true;
    int prev = -1, tc = 0;
    for (int u = cid; u < p.num_units && alive; u += ncl, ++tc) {
      const ConvPhase& ph = find_phase(p, u);
      const bool past = ((u - ph.unit_begin) / p.n_tiles) * kBM + r >= ph.rows;
      for (int kb = 0; kb < ph.num_kb; ++kb) {
        // the stage has landed, and the MMAs that read TMEM stage j before have completed (they run ahead
        // of the copies, so that wait rarely waits)
        const bool ok = wait(&full[s], par, p.err, kSiteFull) && wait(&aempty[j], apar ^ 1, p.err, kSiteEmpty);
        if (!__all_sync(0xffffffffu, ok)) {  // warp-uniform
          alive = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = sbase + s * stage_bytes;
        uint32_t wx[4][4], wd[4][4], o[16];
        dconv_row_load(a0, a0 + a_bytes, r, h, wx, wd);
        if (p.act == 3) dconv_row_half<3>(wx, wd, h, tbl, p.xf_C, kb * D::BKE, past, o);
        else dconv_row_half<2>(wx, wd, h, tbl, p.xf_C, kb * D::BKE, past, o);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // ordered after this warp's reads of the stage (release)
        tmem_st16(tq + static_cast<uint32_t>(j * 32), o);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfull[j]);
        if (++s == S) {
          s = 0;
          par ^= 1;
        }
        if (++j == TA) {
          j = 0;
          apar ^= 1;
        }
      }
      if (alive && prev >= 0 && !epilogue(prev, tc - 1)) alive = false;
      prev = u;
    }
    if (alive && prev >= 0) epilogue(prev, tc - 1);
  } else {
    // ------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    // Epilogue warps: 6-9, or 2-9 for bf16 with the A operand by TMA (the gather warps are free then).
    // Warp w reads TMEM lane quarter w & 3; with eight warps the two warps of a quarter split the
    // tile's 32-column chunks in two halves [cb, ce).
    const int nthr = ep8 ? 256 : 128;
    const int et = threadIdx.x - (kThreads - nthr);  // 0 .. nthr-1 within the epilogue warps
    const int half = ep8 ? (warp - 2) / 4 : 0;
    const int hcols = ep8 ? 32 * ((BN / 32 + 1) / 2) : BN;
    const int cb = half * hcols, ce = half ? BN : hcols;
    T* out = static_cast<T*>(p.out);
    T* out2 = static_cast<T*>(p.out2);
    const bool vec = (p.out_ld % D::EC) == 0;
    // bf16: whole 32-byte stores (a whole sector per lane) when the rows and both outputs start on 32-byte
    // boundaries; fp32 keeps 16-byte stores
    const bool vec32 = DT == 1 && vec && (((static_cast<size_t>(p.out_ld) * sizeof(T)) | reinterpret_cast<uintptr_t>(p.out) |
                                           reinterpret_cast<uintptr_t>(p.out2)) & 31u) == 0;
    // batch-statistics scratch: per-warp column sums and squares, tile means
    float* red = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(tmem_slot) + 16);
    float* red2 = red + 4 * BN;
    float* tmean = red2 + 4 * BN;
    // per-column epilogue constants of the current column tile
    float* sc_s = tmean + BN;
    float* sh_s = sc_s + BN;
    // per-column shift of the statistics pass: epilogue shift minus the statistics shift
    float* kst = sh_s + BN;
    int cur_n_tile = -1;
    // After the first tile, tmean holds the previous tile's column means and
    // serves as the shift of a single-pass (shifted sums) statistic.
    bool have_shift = false;
    // running merge of this CTA's tile statistics, columns et and et + 128
    float cta_n = 0.f, cta_mean0 = 0.f, cta_m20 = 0.f, cta_mean1 = 0.f, cta_m21 = 0.f;
    auto emit = [&](int m_tile, int n_tile, int c, float cnt, float mean, float m2) {
      if (p.stats_per_cta) {
        const float nn = cta_n + cnt, f = cnt / nn;
        if (c < 128) {
          const float d = mean - cta_mean0;
          cta_mean0 = fmaf(d, f, cta_mean0);
          cta_m20 += m2 + d * d * cta_n * f;
        } else {
          const float d = mean - cta_mean1;
          cta_mean1 = fmaf(d, f, cta_mean1);
          cta_m21 += m2 + d * d * cta_n * f;
        }
      } else {
        float* o = p.stats + (static_cast<size_t>(m_tile) * p.N + n_tile * BN + c) * 3;
        o[0] = cnt;
        o[1] = mean;
        o[2] = m2;
      }
    };
    int tc = 0;
    for (int u = cid; u < p.num_units; u += ncl, ++tc) {
      const ConvPhase& ph = find_phase(p, u);
      const int local = u - ph.unit_begin;
      const int m_tile = pair ? 2 * (local / p.n_tiles) + static_cast<int>(rank) : local / p.n_tiles;
      const int n_tile = local % p.n_tiles;
      const int buf = tc % nbuf;
      // lane 0 of each warp waits; the four warps agree before anyone goes on,
      // so the warp-aligned tcgen05.ld and the named barriers below stay
      // uniform even when a wait gives up
      if (n_tile != cur_n_tile) {
        // safe to overwrite: every epilogue thread has passed the previous
        // unit's barrier below, after its last read of these arrays
        for (int c = et; c < BN; c += nthr) {
          const int col = n_tile * BN + c;
          sc_s[c] = (p.ep_scale && col < p.N) ? p.ep_scale[col] : 1.f;
          sh_s[c] = (p.ep_shift && col < p.N) ? p.ep_shift[col] : 0.f;
        }
        cur_n_tile = n_tile;
      }
      int ok = 1;
      if (lane == 0) ok = wait(&tfull[buf], (tc / nbuf) & 1, p.err, kSiteTFull) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!named_bar_and(1, nthr, ok)) break;
      tc_fence_after();
      const int m = m_tile * kBM + row;
      const bool valid = m < ph.rows;
      size_t obase = 0;
      int oh_px = 0, ow_px = 0;  // output pixel of the row
      if (valid) {
        const int n = static_cast<int>(fdiv(static_cast<uint32_t>(m), ph.div_HaWa));
        const int rem = m - n * ph.Ha * ph.Wa;
        const int a = static_cast<int>(fdiv(static_cast<uint32_t>(rem), ph.div_Wa));
        const int b = rem - a * ph.Wa;
        oh_px = ph.oh0 + a * p.os;
        ow_px = ph.ow0 + b * p.os;
        obase = (static_cast<size_t>(n * p.Ho + oh_px) * p.Wo + ow_px) * p.out_ld;
      }
      // layer-norm partials of this row over the half's columns: exact two-pass per 32 columns, merged
      // across the chunks with Chan's formula (the chunks before column cc hold cc - cb values)
      float rmean = 0.f, rm2 = 0.f;
      const bool zero = ph.num_kb == 0;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * tcs;
      // A in TMEM: each chunk's two halves (hi x hi + lo x hi, then hi x lo). One chunk and no statistics
      // pass (which reads the accumulator again): the halves are added in registers below; else they are
      // summed into the first block in TMEM
      const bool ts_sum = ts && !zero && !p.stats && ph.num_kb <= kpc;
      if (ts && !zero && !ts_sum)
        fold_chunks(taddr, BN, 2 * ((ph.num_kb + kpc - 1) / kpc), cb, ce);
      else if (DT == 0 && ph.num_kb > kpc)  // several accumulator chunks: summed into the first
        fold_chunks(taddr, BN, (ph.num_kb + kpc - 1) / kpc, cb, ce);
      // columns are read from TMEM 64 at a time (two 32-column loads, one wait)
      auto fetch = [&](int c0, uint32_t (&ra)[32], uint32_t (&rb)[32]) {
        const int c1 = c0 + 32 < ce ? c0 + 32 : c0;
        tmem_ld32(taddr + c0, ra);
        tmem_ld32(taddr + c1, rb);
        tmem_ld_wait2(ra, rb);
      };
      auto pass1 = [&](int cc, const uint32_t (&r)[32]) {
        const int col0 = n_tile * BN + cc;
        const int ncols = p.N - col0;
        if (ncols <= 0) return;  // uniform across the warp
        // column constants and shifts are read as 16-byte vectors (the tensor core's operand reads
        // already use most of the shared-memory bandwidth)
        float v[32];
        ep_columns(r, zero, p.ep_scale != nullptr, sc_s + cc, sh_s + cc, v);
        if (valid && p.seg) {
          store_phase_runs<T>(out, obase, oh_px, ow_px, col0, v, ncols, p);
        } else if (valid && !p.out_act && !p.rstats && !out2) {
          store_row32<T>(out + obase + col0, v, ncols, vec, vec32);  // one rounding to T
        } else if (valid) {
          float o[32];
          if constexpr (DT == 0) {  // fp32: the activation dispatched once per segment (see act_row32)
            if (p.out_act) {
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = v[e];
              act_row32<false>(p.act, o);
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = to_stored<T>(v[e]);
            }
          } else {  // bf16: the fast activations are single instructions
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = p.out_act ? act_f(p.act, v[e], true) : to_stored<T>(v[e]);
          }
          if (p.rstats) {  // o holds the stored value (the host never combines rstats with out_act)
            const int nc = ncols < 32 ? ncols : 32;
            float sum = 0.f;
#pragma unroll
            for (int e = 0; e < 32; ++e) sum += e < nc ? o[e] : 0.f;
            const float fnc = static_cast<float>(nc), cm = sum / fnc;
            float m2 = 0.f;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const float d = e < nc ? o[e] - cm : 0.f;
              m2 = fmaf(d, d, m2);
            }
            const float rn = static_cast<float>(cc - cb), nn = rn + fnc, dl = cm - rmean, f = fnc / nn;
            rmean = fmaf(dl, f, rmean);
            rm2 += m2 + dl * dl * rn * f;
          }
          store_row32<T>(out + obase + col0, o, ncols, vec, vec32);
          if (out2) {
            if constexpr (DT == 0) {
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = to_stored<T>(v[e]);
              act_row32<false>(p.act, o);
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = act_f(p.act, to_stored<T>(v[e]), true);
            }
            store_row32<T>(out2 + obase + col0, o, ncols, vec, vec32);
          }
        }
      };
      // 64 columns per step (32 with ts_sum: columns c0 .. c0 + 31 of both halves, added)
      for (int c0 = cb; c0 < ce; c0 += ts_sum ? 32 : 64) {
        uint32_t ra[32], rb[32];
        if (ts_sum) {
          tmem_ld32(taddr + c0, ra);
          tmem_ld32(taddr + static_cast<uint32_t>(BN + c0), rb);
          tmem_ld_wait2(ra, rb);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 v2 = __fadd2_rn(f2(ra[e], ra[e + 1]), f2(rb[e], rb[e + 1]));
            ra[e] = __float_as_uint(v2.x);
            ra[e + 1] = __float_as_uint(v2.y);
          }
        } else {
          fetch(c0, ra, rb);
        }
        pass1(c0, ra);
        if (!ts_sum && c0 + 32 < ce) pass1(c0 + 32, rb);
      }
      if (p.rstats && valid) {
        const int nh = ep8 ? 2 : 1;
        float* o = p.rstats + ((obase / p.out_ld * p.n_tiles + n_tile) * nh + half) * 2;
        o[0] = rmean;
        o[1] = rm2;
      }
      if (p.stats) {
        // Statistics of the unrounded value v, from a second read of the accumulator
        // (colstats32): shifted sums d = v - s give mean = s + sum(d)/n and
        // M2 = sum(d^2) - sum(d)^2/n. After the first tile s is the previous tile's
        // column mean; the first tile takes its own mean from a plain pass first.
        const int cnt = min(kBM, ph.rows - m_tile * kBM);
        const int cols = min(BN, p.N - n_tile * BN);
        const float fc = static_cast<float>(cnt);
        const int qrows = cnt - q * 32;  // valid rows of this warp's lane quarter
        unsigned rowmask = 0u;
#pragma unroll
        for (int i = 0; i < 4; ++i) rowmask |= ((lane >> 2) + 8 * i >= qrows ? 1u : 0u) << i;
        const float* av = p.ep_scale ? sc_s : nullptr;
        const uint32_t tq = taddr;
        // pass 0 (first tile only): plain sums for the tile's own mean; pass 1: shifted sums
#pragma unroll 1
        for (int pass = have_shift ? 1 : 0; pass < 2; ++pass) {
          const float* kc = pass ? kst : sh_s;
          for (int cc = cb; cc < ce && cc < cols; cc += 32)
            colstats32(tq + cc, zero, av ? av + cc : nullptr, kc + cc, rowmask, lane, red + q * BN + cc,
                       red2 + q * BN + cc);
          named_bar_sync(1, nthr);
          if (pass == 0) {
            for (int c = et; c < BN; c += nthr) {
              const float m = c < cols ? (red[c] + red[BN + c] + red[2 * BN + c] + red[3 * BN + c]) / fc : 0.f;
              tmean[c] = m;
              kst[c] = sh_s[c] - m;
            }
            named_bar_sync(1, nthr);
          }
        }
        for (int c = et; c < cols; c += nthr) {
          const float s1 = red[c] + red[BN + c] + red[2 * BN + c] + red[3 * BN + c];
          const float s2 = red2[c] + red2[BN + c] + red2[2 * BN + c] + red2[3 * BN + c];
          const float mean = tmean[c] + s1 / fc;
          emit(m_tile, n_tile, c, fc, mean, fmaxf(s2 - s1 * (s1 / fc), 0.f));
          // the next tile's shift (read after the next unit's barrier; used when the
          // column tile stays the same)
          tmean[c] = mean;
          kst[c] = sh_s[c] - mean;
        }
        cta_n += fc;
        have_shift = p.n_tiles == 1;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (pair && !leader) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[buf]), 0));
        else mbar_arrive(&tempty[buf]);
      }
    }
    if (p.stats && p.stats_per_cta) {
      for (int c = et; c < min(BN, p.N); c += nthr) {
        float* o = p.stats + (static_cast<size_t>(blockIdx.x) * p.N + c) * 3;
        o[0] = cta_n;
        o[1] = c < 128 ? cta_mean0 : cta_mean1;
        o[2] = c < 128 ? cta_m20 : cta_m21;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (pair) cluster_sync();  // no remote arrival or MMA write into this CTA is still in flight
  if (warp == 1) {
    tc_fence_after();
    if (pair) tmem_dealloc_pair(tmem_base, tcols);
    else tmem_dealloc(tmem_base, tcols);
  }
}

// --------------------------------------------------------------------------
// wgrad: D[k][oc] = sum over a split of the pixels of im2col(X)[pix][k] *
// d_conv[pix][oc]; written as fp32 partials [split][oc][k].
// --------------------------------------------------------------------------
// PAIR: CTA pairs (cta_group::2): the pair computes 256 rows of dW (two m-tiles); each CTA holds its
// 128 rows of A and half of the d_conv columns (BN a multiple of 128).
template <int DT, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1) wgrad_gemm_kernel(const __grid_constant__ WgradParams p) {
  pdl_entry();
  using D = Dt<DT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int BN = p.BN;
  constexpr bool pair = PAIR;
  static_assert(!PAIR || DT == 1, "CTA pairs run bf16 only");
  const uint32_t a_bytes = kBM * 128, b_bytes = BN * 128;
  const uint32_t b_own = pair ? b_bytes / 2 : b_bytes;  // a pair member holds half of the oc columns
  // fp32 with A in TMEM (WgradParams::ts): a stage holds the d_conv hi and lo rows only
  const bool ts = DT == 0 && p.ts;
  // d_conv formed from the pre-activation and dY boxes (WgradParams::xf): a stage holds X, then both
  const bool xf = DT == 1 && !PAIR && p.xf;
  const uint32_t stage_bytes = ts ? 2 * b_bytes
                                  : (xf ? a_bytes + 2 * b_bytes
                                        : D::NS * (a_bytes + b_own) * (DT == 1 && p.kps > 1 ? p.kps : 1));
  const int S = p.stages;
  const int KPS = DT == 1 && p.kps > 1 ? p.kps : 1;  // k-blocks per stage (bf16 with A by TMA)
  const uint32_t panel = 8192u * KPS;                  // distance between MN-major panels / d_conv boxes
  // fp32 with X by TMA: a ring of raw tiles (X chunks then d_conv chunks, 32 pixel rows x 128 B each)
  const bool raw_a = DT == 0 && p.a_tma;
  const int NR = raw_a ? p.rstages : 0;
  const uint32_t raw_bytes = a_bytes + b_bytes;
  uint8_t* rawp = smem + S * stage_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(rawp + NR * raw_bytes);
  uint64_t* empty = full + kMaxStages;
  uint64_t* tfull = empty + kMaxStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* rfull = tempty + 2;
  uint64_t* rempty = rfull + kMaxStages;
  uint64_t* sfull = rempty + kMaxStages;  // xf: d_conv formed in the stage
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sfull + kMaxStages);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t rbase = smem_u32(rawp);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // two accumulators (2 * BN columns each with A in TMEM), then one TMEM stage of A per stage (hi: 32
  // columns, lo: 32)
  const int acols = ts ? 2 * BN : BN;
  const uint32_t tcols = tmem_cols_for(2 * acols + (ts ? S * 64 : 0));
  const uint32_t ta0 = static_cast<uint32_t>(2 * acols);
  constexpr int KP = (DT == 1) ? 64 : 32;  // pixels per k-block
  const uint32_t rank = pair ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const int cid = pair ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int ncl = pair ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      // the TMA thread and/or one per producer warp (fp32 raw tiles: one per transposing warp, 2-9)
      mbar_init(&full[s], DT == 1 ? (p.a_tma ? 1 : 4 + 1) : (raw_a ? 8 : 4));
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      // epilogue warps (of both CTAs when paired; xf and fp32 raw tiles: warps 2-9)
      mbar_init(&tempty[b], (pair || xf || raw_a) ? 8 : 4);
    }
    for (int r = 0; r < NR; ++r) {
      mbar_init(&rfull[r], 1);   // the TMA thread
      mbar_init(&rempty[r], 8);  // one arrival per transposing warp (2-9)
    }
    if (xf)
      for (int s = 0; s < S; ++s) mbar_init(&sfull[s], 8);  // one arrival per transforming warp
    fence_mbar_init();
    if (DT == 1 || raw_a) tma_prefetch_desc(&p.tmap_dc);
    if (p.a_tma) tma_prefetch_desc(&p.tmap_x);
    if (xf) tma_prefetch_desc(&p.tmap_dy);
  }
  if (warp == 1) {
    if (pair) {
      tmem_alloc_pair(tmem_slot, tcols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, tcols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (pair) cluster_sync();  // the peer's barriers are initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  auto decode = [&](int u, int& m_tile, int& n_tile, int& kb0, int& kb1) {
    m_tile = pair ? 2 * (u % p.m_tiles) + static_cast<int>(rank) : u % p.m_tiles;
    const int rest = u / p.m_tiles;
    n_tile = rest % p.n_tiles;
    const int split = rest / p.n_tiles;
    kb0 = split * p.kb_per_split;
    kb1 = min(p.kb_total, kb0 + p.kb_per_split);
  };

  if (warp == 0) {
    // ------------------------------------------------ B producer (bf16: TMA of d_conv)
    if (DT == 1 && lane == 0) {
      int s = 0;
      uint32_t par = 0;
      bool alive = true;
      for (int u = cid; u < p.num_units && alive; u += ncl) {
        int m_tile, n_tile, kb0, kb1;
        decode(u, m_tile, n_tile, kb0, kb1);
        // A panels (64 k-rows each): tap offsets and channel of each panel
        int pc[2], pkw[2], pkh[2];
        uint32_t a_tx = 0;
        if (p.a_tma) {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int kc = m_tile * kBM + 64 * j;
            const int tap = static_cast<int>(fdiv(static_cast<uint32_t>(kc), p.div_Cs));
            pkh[j] = static_cast<int>(fdiv(static_cast<uint32_t>(tap), p.div_KW));
            pkw[j] = tap - pkh[j] * p.KW;
            pc[j] = kc < p.Mk ? kc - tap * p.Cs : -1;  // -1: k padding, panel not loaded (its rows are discarded)
            if (pc[j] >= 0) a_tx += 8192;
          }
        }
        if (pair) {
          // the even CTA's barrier expects both members' panels: add the peer's loaded panels
          const int peer = m_tile ^ 1;
#pragma unroll
          for (int j = 0; j < 2; ++j)
            if (peer * kBM + 64 * j < p.Mk) a_tx += 8192;
        }
        for (int g0 = kb0; g0 < kb1; g0 += KPS) {  // one stage: k-blocks g0 .. g0 + KPS - 1 (copies cover all)
          if (!wait(&empty[s], par ^ 1, p.err, kSiteEmpty)) {
            alive = false;
            break;
          }
          const uint32_t a0 = sbase + s * stage_bytes;
          const uint32_t b0 = a0 + KPS * a_bytes;
          const int pix = g0 * KP;  // first pixel of the stage; the maps walk the next KPS * KP
          if (pair) {
            const uint32_t bar = mapa_shared(smem_u32(&full[s]), 0);
            if (leader) mbar_arrive_expect_tx(&full[s], KPS * (b_bytes + a_tx));
            const int n = static_cast<int>(fdiv(static_cast<uint32_t>(pix), p.div_OHOW));
            const int rem = pix - n * p.OH * p.OW;
            const int oh = static_cast<int>(fdiv(static_cast<uint32_t>(rem), p.div_OW));
            const int ow = rem - oh * p.OW;
#pragma unroll
            for (int j = 0; j < 2; ++j)
              if (pc[j] >= 0)
                tma_load_im2col_4d_pair(a0 + j * panel, &p.tmap_x, bar, pc[j], ow * p.S - p.P, oh * p.S - p.P, n,
                                        static_cast<uint16_t>(pkw[j]), static_cast<uint16_t>(pkh[j]));
            const int nb = BN / 128;  // this member's 64-column boxes
            for (int jn = 0; jn < nb; ++jn)
              tma_load_2d_pair(b0 + jn * panel, &p.tmap_dc, bar,
                               n_tile * BN + 64 * (static_cast<int>(rank) * nb + jn), pix);
          } else if (xf) {
            // 1x1, stride 1: X, the pre-activation and dY are [n_pix][channels] matrices; each comes as one
            // copy of its 64-pixel panels (a 3-D view: 64 channels x pixels x 64-channel groups)
            mbar_arrive_expect_tx(&full[s], a_bytes + 2 * b_bytes);
            tma_load_3d(a0, &p.tmap_x, &full[s], 0, pix, 2 * m_tile);
            tma_load_3d(b0, &p.tmap_dc, &full[s], 0, pix, n_tile * (BN / 64));
            tma_load_3d(b0 + b_bytes, &p.tmap_dy, &full[s], 0, pix, n_tile * (BN / 64));
          } else {
            mbar_arrive_expect_tx(&full[s], KPS * (b_bytes + a_tx));
            if (p.a_tma) {
              const int n = static_cast<int>(fdiv(static_cast<uint32_t>(pix), p.div_OHOW));
              const int rem = pix - n * p.OH * p.OW;
              const int oh = static_cast<int>(fdiv(static_cast<uint32_t>(rem), p.div_OW));
              const int ow = rem - oh * p.OW;
#pragma unroll
              for (int j = 0; j < 2; ++j)
                if (pc[j] >= 0)
                  tma_load_im2col_4d(a0 + j * panel, &p.tmap_x, &full[s], pc[j], ow * p.S - p.P, oh * p.S - p.P, n,
                                     static_cast<uint16_t>(pkw[j]), static_cast<uint16_t>(pkh[j]));
            }
            for (int jn = 0; jn < BN / 64; ++jn)
              tma_load_2d(b0 + jn * panel, &p.tmap_dc, &full[s], n_tile * BN + 64 * jn, pix);
          }
          if (++s == S) {
            s = 0;
            par ^= 1;
          }
        }
      }
      if (pair) {
        // the even CTA's commits land in this CTA's empty barriers: let every stage's last use finish
        for (int i = 0; i < S && alive; ++i) {
          if (!wait(&empty[s], par ^ 1, p.err, kSiteEmpty)) break;
          if (++s == S) {
            s = 0;
            par ^= 1;
          }
        }
      }
    }
    if (raw_a && lane == 0) {
      // ------------------------------------------------ fp32: raw X and d_conv tiles by TMA
      int r = 0;
      uint32_t rpar = 0;
      bool alive = true;
      for (int u = cid; u < p.num_units && alive; u += ncl) {
        int m_tile, n_tile, kb0, kb1;
        decode(u, m_tile, n_tile, kb0, kb1);
        // X chunks: 32 k-rows (one tap, 32 channels) each; past Mk not loaded (those rows are discarded)
        int pc[4], pkw[4], pkh[4];
        uint32_t tx = static_cast<uint32_t>(BN / 32) * 4096u;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int kc = m_tile * kBM + 32 * c;
          const int tap = static_cast<int>(fdiv(static_cast<uint32_t>(kc), p.div_Cs));
          pkh[c] = static_cast<int>(fdiv(static_cast<uint32_t>(tap), p.div_KW));
          pkw[c] = tap - pkh[c] * p.KW;
          pc[c] = kc < p.Mk ? kc - tap * p.Cs : -1;
          if (pc[c] >= 0) tx += 4096u;
        }
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!wait(&rempty[r], rpar ^ 1, p.err, kSiteEmpty)) {
            alive = false;
            break;
          }
          const uint32_t r0 = rbase + r * raw_bytes;
          mbar_arrive_expect_tx(&rfull[r], tx);
          const int pix = kb * KP;  // first pixel of the k-block; the maps walk the next 32
          const int n = static_cast<int>(fdiv(static_cast<uint32_t>(pix), p.div_OHOW));
          const int rem = pix - n * p.OH * p.OW;
          const int oh = static_cast<int>(fdiv(static_cast<uint32_t>(rem), p.div_OW));
          const int ow = rem - oh * p.OW;
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (pc[c] >= 0)
              tma_load_im2col_4d(r0 + c * 4096, &p.tmap_x, &rfull[r], pc[c], ow * p.S - p.P, oh * p.S - p.P, n,
                                 static_cast<uint16_t>(pkw[c]), static_cast<uint16_t>(pkh[c]));
          for (int jn = 0; jn < BN / 32; ++jn)
            tma_load_2d(r0 + a_bytes + jn * 4096, &p.tmap_dc, &rfull[r], n_tile * BN + 32 * jn, pix);
          if (++r == NR) {
            r = 0;
            rpar ^= 1;
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      const uint32_t idesc = idesc_f32acc(pair ? 2 * kBM : kBM, BN, D::FMT, DT == 1, DT == 1);
      const uint32_t idesc2 = idesc_f32acc(kBM, 2 * BN, D::FMT, false, false);  // A_hi x [B_hi; B_lo]
      int s = 0;
      uint32_t par = 0;
      int tc = 0;
      bool alive = true;
      for (int u = cid; u < p.num_units && alive; u += ncl, ++tc) {
        int m_tile, n_tile, kb0, kb1;
        decode(u, m_tile, n_tile, kb0, kb1);
        const int buf = tc & 1;
        if (!wait(&tempty[buf], ((tc >> 1) & 1) ^ 1, p.err, kSiteTEmpty)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + buf * acols;
        for (int g0 = kb0; g0 < kb1; g0 += KPS) {  // one stage: k-blocks g0 .. g0 + nk - 1
          const int nk = min(KPS, kb1 - g0);
          if (!wait(xf ? &sfull[s] : &full[s], par, p.err, kSiteFull)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sbase + s * stage_bytes;
          const uint32_t b0 = ts ? a0 : a0 + D::NS * a_bytes * KPS;
          const uint32_t ah = tmem_base + ta0 + static_cast<uint32_t>(s * 64);
#pragma unroll
          for (int i = 0; i < kMaxKps; ++i) {
            if (i >= nk) break;
            const int kb = g0 + i;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint32_t acc = (kb > kb0 || kk) ? 1u : 0u;
              if (ts) {
                const uint64_t bd = sdesc_sw128(b0 + kk * 32, 16, 1024);  // 2 BN rows: hi, then lo
                mma_tf32_ta(d, ah + kk * 8, bd, idesc2, acc);
                mma_tf32_ta(d, ah + 32 + kk * 8, bd, idesc, 1u);
              } else if (DT == 1) {
                // MN-major: 16 pixel rows per MMA (2048 B) of k-block i (8 KB * i into each panel), panels of
                // 64 k / 64 oc `panel` bytes apart
                const uint64_t ad = sdesc_sw128(a0 + i * 8192 + kk * 2048, panel, 1024);
                const uint64_t bd = sdesc_sw128(b0 + i * 8192 + kk * 2048, panel, 1024);
                if (pair) mma_bf16_pair(d, ad, bd, idesc, acc);
                else mma_bf16(d, ad, bd, idesc, acc);
              } else {
                const uint64_t ad = sdesc_sw128(a0 + kk * 32, 16, 1024);
                const uint64_t bd = sdesc_sw128(b0 + kk * 32, 16, 1024);
                const uint64_t al = sdesc_sw128(a0 + a_bytes + kk * 32, 16, 1024);
                const uint64_t bl = sdesc_sw128(b0 + b_bytes + kk * 32, 16, 1024);
                mma_tf32(d, al, bd, idesc, acc);
                mma_tf32(d, ad, bl, idesc, 1u);
                mma_tf32(d, ad, bd, idesc, 1u);
              }
            }
          }
          if (pair) mma_commit_pair(&empty[s]);
          else mma_commit(&empty[s]);
          if (++s == S) {
            s = 0;
            par ^= 1;
          }
        }
        if (alive) {
          if (pair) mma_commit_pair(&tfull[buf]);
          else mma_commit(&tfull[buf]);
        }
      }
    }
  } else if (xf) {
    // ------------------------------------------------ d_conv from the pre-activation and dY panels, and the epilogue
    // Warps 2-9 turn each landed stage's pre-activation panels into d_conv (two rows of every panel per thread;
    // the MMA waits for sfull); after a unit's k-blocks they write the unit before it (its accumulator
    // completed meanwhile): two warps per TMEM lane quarter, one per column half. The terms of d_conv follow
    // the TMEM slot.
    const int t = threadIdx.x - 64;
    float* tbl = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(tmem_slot) + 16);
    load_xform_terms(tbl, p.xf_tbl, p.xf_C, t, 256);
    const int q = warp & 3, half = (warp - 2) >> 2;
    const int hcols = 32 * ((BN / 32 + 1) / 2);
    const int cb = half * hcols, ce = half ? BN : hcols;
    auto epilogue = [&](int u, int tc) -> bool {
      int m_tile, n_tile, kb0, kb1;
      decode(u, m_tile, n_tile, kb0, kb1);
      const int split = u / (p.m_tiles * p.n_tiles);
      const int buf = tc & 1;
      int ok = 1;
      if (lane == 0) ok = wait(&tfull[buf], (tc >> 1) & 1, p.err, kSiteTFull) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
      tc_fence_after();
      const int m = m_tile * kBM + q * 32 + lane;
      const bool zero = kb1 <= kb0;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * acols;
      for (int c0 = cb; c0 < ce; c0 += 32) {
        if (n_tile * BN + c0 >= p.N) break;  // uniform across the warp
        uint32_t r[32];
        tmem_ld32(taddr + c0, r);
        tmem_ld_wait32(r);
        if (m < p.Mk) {
          float* dst = p.partial + (static_cast<size_t>(split) * p.N + n_tile * BN + c0) * p.Mk + m;
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (n_tile * BN + c0 + e < p.N) dst[static_cast<size_t>(e) * p.Mk] = zero ? 0.f : __uint_as_float(r[e]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
      return true;
    };
    int s = 0;
    uint32_t par = 0;
    bool alive = true;
    int prev = -1, tc = 0;
    for (int u = cid; u < p.num_units && alive; u += ncl, ++tc) {
      int m_tile, n_tile, kb0, kb1;
      decode(u, m_tile, n_tile, kb0, kb1);
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!__all_sync(0xffffffffu, wait(&full[s], par, p.err, kSiteFull))) {  // warp-uniform
          alive = false;
          break;
        }
        const uint32_t b0 = sbase + s * stage_bytes + a_bytes;
        if (p.act == 3)
          dconv_xform<3, KP / 32, 32>(b0, b0 + b_bytes, BN / 64, tbl, p.xf_C, n_tile * BN, p.n_pix - kb * KP, t);
        else
          dconv_xform<2, KP / 32, 32>(b0, b0 + b_bytes, BN / 64, tbl, p.xf_C, n_tile * BN, p.n_pix - kb * KP, t);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfull[s]);
        if (++s == S) {
          s = 0;
          par ^= 1;
        }
      }
      if (alive && prev >= 0 && !epilogue(prev, tc - 1)) alive = false;
      prev = u;
    }
    if (alive && prev >= 0) epilogue(prev, tc - 1);
  } else if (raw_a) {
    // ------------------------------------------------ fp32: transpose the raw tiles into tf32 hi / lo, and the epilogue
    // Warps 2-9. A raw chunk is 32 pixel rows x 32 channels (128-byte swizzle as the TMA wrote it); the stage
    // wants K-major rows of 32 pixels per channel. A half-chunk transpose: lane (pq, cq) reads the 4 x 4 block
    // of pixels 4pq.. and channels 4cq.. (four 16-byte reads), splits it and writes four channel rows of four
    // pixels to the hi and lo tiles (both sides spread over all banks); warps 2-5 take them in turn.
    // With A in TMEM (ts) the X chunks go to TMEM instead: warp w moves pixels 16h .. 16h + 15 (h = 0 for
    // warps 2-5, 1 for warps 6-9) of X chunk w & 3 (its TMEM lane quarter), lane ch reading channel ch, and
    // stores hi / lo into columns 16h.. / 32 + 16h.. of the stage's TMEM rows (column = pixel = k); the
    // half-chunk transposes cover the d_conv chunks only. After a unit's k-blocks the eight warps write the
    // unit before it (its accumulator completed meanwhile), one column half each.
    const int wi = warp - 2;
    const int q = warp & 3, half = wi >> 2;
    const int pq = lane & 7, cql = lane >> 3;
    const int hcols = 32 * ((BN / 32 + 1) / 2);
    const int cb = half * hcols, ce = half ? BN : hcols;
    auto epilogue = [&](int u, int tcu) -> bool {
      int m_tile, n_tile, kb0, kb1;
      decode(u, m_tile, n_tile, kb0, kb1);
      const int split = u / (p.m_tiles * p.n_tiles);
      const int buf = tcu & 1;
      int ok = 1;
      if (lane == 0) ok = wait(&tfull[buf], (tcu >> 1) & 1, p.err, kSiteTFull) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, ok, 0)) return false;
      tc_fence_after();
      const int m = m_tile * kBM + q * 32 + lane;
      const bool zero = kb1 <= kb0;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * acols;
      for (int c0 = cb; c0 < ce; c0 += 32) {
        if (n_tile * BN + c0 >= p.N) break;  // uniform across the warp
        uint32_t ra[32], rb[32];
        tmem_ld32(taddr + c0, ra);
        if (ts) {  // column c holds hi x hi + lo x hi, column BN + c hi x lo
          tmem_ld32(taddr + BN + c0, rb);
          tmem_ld_wait2(ra, rb);
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 v2 = __fadd2_rn(f2(ra[e], ra[e + 1]), f2(rb[e], rb[e + 1]));
            ra[e] = __float_as_uint(v2.x);
            ra[e + 1] = __float_as_uint(v2.y);
          }
        } else {
          tmem_ld_wait32(ra);
        }
        if (m < p.Mk) {
          float* dst = p.partial + (static_cast<size_t>(split) * p.N + n_tile * BN + c0) * p.Mk + m;
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (n_tile * BN + c0 + e < p.N) dst[static_cast<size_t>(e) * p.Mk] = zero ? 0.f : __uint_as_float(ra[e]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
      return true;
    };
    int r = 0, s = 0;
    uint32_t rpar = 0, par = 0;
    bool alive = true;
    int prev = -1, tc = 0;
    const int nchunk = ts ? BN / 32 : 4 + BN / 32;
    for (int u = cid; u < p.num_units && alive; u += ncl, ++tc) {
      int m_tile, n_tile, kb0, kb1;
      decode(u, m_tile, n_tile, kb0, kb1);
      (void)n_tile;
      const int nvalid = min(4, (p.Mk - m_tile * kBM + 31) / 32);  // X chunks inside Mk
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!__all_sync(0xffffffffu, wait(&rfull[r], rpar, p.err, kSiteFull) &&
                                         wait(&empty[s], par ^ 1, p.err, kSiteEmpty))) {  // warp-uniform
          alive = false;
          break;
        }
        const uint32_t r0 = rbase + r * raw_bytes;
        const uint32_t a0 = sbase + s * stage_bytes;
        const uint32_t b0 = ts ? a0 : a0 + 2 * a_bytes;
        if (ts) {
          tc_fence_after();  // the MMAs that read this TMEM stage have completed (empty[s])
          if (q < nvalid) {  // rows past Mk keep stale values: their dW rows are discarded
            const uint32_t src = r0 + q * 4096 + (lane & 3) * 4;
            const uint32_t dst = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + ta0 + s * 64;
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
              const int px = 16 * half + e;
              uint32_t x, y;
              asm volatile("ld.shared.b32 %0, [%1];"
                           : "=r"(x)
                           : "r"(src + px * 128 + ((((lane >> 2) ^ (px & 7))) << 4)));
              asm volatile("ld.shared.b32 %0, [%1];"
                           : "=r"(y)
                           : "r"(src + (px + 1) * 128 + ((((lane >> 2) ^ ((px + 1) & 7))) << 4)));
              split_tf32x2(__uint_as_float(x), __uint_as_float(y), hi[e], lo[e], hi[e + 1], lo[e + 1]);
            }
            tmem_st16(dst + 16 * half, hi);
            tmem_st16(dst + 32 + 16 * half, lo);
            tmem_st_wait();
          }
        }
        for (int it = wi; it < 2 * nchunk; it += 4) {
          if (half) break;  // the half-chunk transposes: warps 2-5
          const int c = ts ? 4 + (it >> 1) : it >> 1;
          if (c < 4 && c >= nvalid) continue;  // uniform across the warp
          const int cq = cql + 4 * (it & 1);
          const bool isa = c < 4;
          const uint32_t src = r0 + c * 4096;  // X chunks 0-3, then d_conv chunks
          const uint32_t hi = isa ? a0 + c * 4096 : b0 + (c - 4) * 4096;
          const uint32_t lo_off = isa ? a_bytes : b_bytes;
          float v[4][4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int px = 4 * pq + i;
            uint32_t x0, x1, x2, x3;
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                         : "r"(src + px * 128 + ((cq ^ (px & 7)) << 4)));
            v[i][0] = __uint_as_float(x0);
            v[i][1] = __uint_as_float(x1);
            v[i][2] = __uint_as_float(x2);
            v[i][3] = __uint_as_float(x3);
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int row = 4 * cq + e;  // channel row within the chunk (the chunk starts on an 8-row atom)
            const uint32_t addr = hi + row * 128 + ((pq ^ (row & 7)) << 4);
            uint32_t h[4], l[4];
#pragma unroll
            for (int i = 0; i < 4; i += 2) split_tf32x2(v[i][e], v[i + 1][e], h[i], l[i], h[i + 1], l[i + 1]);
            st_shared_v4(addr, h[0], h[1], h[2], h[3]);
            st_shared_v4(addr + lo_off, l[0], l[1], l[2], l[3]);
          }
        }
        if (ts) tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&full[s]);
          mbar_arrive(&rempty[r]);
        }
        if (++r == NR) {
          r = 0;
          rpar ^= 1;
        }
        if (++s == S) {
          s = 0;
          par ^= 1;
        }
      }
      if (alive && prev >= 0 && !epilogue(prev, tc - 1)) alive = false;
      prev = u;
    }
    if (alive && prev >= 0) epilogue(prev, tc - 1);
  } else if (warp < 6) {
    const int t = threadIdx.x - 64;
    const char* xs = static_cast<const char*>(p.x);
    int s = 0;
    uint32_t par = 0;
    int it = 0;
    bool alive = true;
    if (DT == 1) {
      // ------------------------------------------------ A producer, bf16, MN-major
      // smem A: two panels (k 0-63, 64-127) of [64 pixel rows][128 B]. Thread
      // pair (2r, 2r+1) owns pixel row r and copies its 16-byte chunks
      // q = 2j + (t & 1), j = 0..7: adjacent lanes read adjacent chunks.
      const int r = t >> 1, half = t & 1;
      if (p.a_tma) alive = false;  // A comes by TMA im2col: nothing to gather
      for (int u = blockIdx.x; u < p.num_units && alive; u += gridDim.x) {
        int m_tile, n_tile, kb0, kb1;
        decode(u, m_tile, n_tile, kb0, kb1);
        int dh[8], dw[8], cofs[8];
        uint32_t dsto[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int q = 2 * j + half;
          const int kc = m_tile * kBM + q * 8;
          const int tap = static_cast<int>(fdiv(static_cast<uint32_t>(kc), p.div_Cs));
          const int kh = static_cast<int>(fdiv(static_cast<uint32_t>(tap), p.div_KW));
          cofs[j] = kc - tap * p.Cs;
          dh[j] = kc < p.Mk ? kh - p.P : -(1 << 28);  // k padding rows read as zero
          dw[j] = (tap - kh * p.KW) - p.P;
          dsto[j] = static_cast<uint32_t>((q >> 3) * 8192 + r * 128 + (((q & 7) ^ (r & 7)) << 4));
        }
        for (int kb = kb0; kb < kb1; ++kb) {
          const int pix = kb * KP + r;
          const bool okp = pix < p.n_pix;
          int n = 0, oh = 0, ow = 0;
          if (okp) {
            n = static_cast<int>(fdiv(static_cast<uint32_t>(pix), p.div_OHOW));
            const int rem = pix - n * p.OH * p.OW;
            oh = static_cast<int>(fdiv(static_cast<uint32_t>(rem), p.div_OW));
            ow = rem - oh * p.OW;
          }
          const int ih0 = oh * p.S, iw0 = ow * p.S;
          const size_t img = static_cast<size_t>(n) * p.H;
          if (!__all_sync(0xffffffffu, wait(&empty[s], par ^ 1, p.err, kSiteEmpty))) {  // warp-uniform
            alive = false;
            break;
          }
          const uint32_t a0 = sbase + s * stage_bytes;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int ih = ih0 + dh[j], iw = iw0 + dw[j];
            const bool ok = okp && static_cast<unsigned>(ih) < static_cast<unsigned>(p.H) &&
                            static_cast<unsigned>(iw) < static_cast<unsigned>(p.W);
            const size_t off = ok ? (((img + ih) * p.W + iw) * p.Cs + cofs[j]) * 2 : 0;
            cp_async16(a0 + dsto[j], xs + off, ok ? 16u : 0u);
          }
          cp_async_commit();
          if (it >= kLag) {
            cp_async_wait<kLag>();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[(it - kLag) % S]);
          }
          ++it;
          if (++s == S) {
            s = 0;
            par ^= 1;
          }
        }
      }
      cp_async_wait<0>();
      fence_proxy_async_smem();
      __syncwarp();
      if (alive && lane == 0)
        for (int q2 = (it > kLag ? it - kLag : 0); q2 < it; ++q2) mbar_arrive(&full[q2 % S]);
    } else {
      // ------------------------------------------------ A and B producers, fp32 -> tf32 hi/lo, K-major
      // A smem rows: k (128), 32 pixel columns; B smem rows: oc (BN), 32 pixel columns.
      const int pc = t & 31, g0 = t >> 5;
      const uint32_t colsw = static_cast<uint32_t>(pc & 3) * 4;
      for (int u = blockIdx.x; u < p.num_units && alive; u += gridDim.x) {
        int m_tile, n_tile, kb0, kb1;
        decode(u, m_tile, n_tile, kb0, kb1);
        int dhs[8], dws[8], cs[8];
        bool oks[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int kc = m_tile * kBM + 4 * (g0 + 4 * i);
          oks[i] = kc < p.Mk;
          const int tap = static_cast<int>(fdiv(static_cast<uint32_t>(kc), p.div_Cs));
          cs[i] = kc - tap * p.Cs;
          const int kh = static_cast<int>(fdiv(static_cast<uint32_t>(tap), p.div_KW));
          dhs[i] = kh - p.P;
          dws[i] = (tap - kh * p.KW) - p.P;
        }
        // the X loads of k-block kb + 1 are issued before k-block kb is split and stored, and the d_conv
        // loads of k-block kb before its X values are, so that their latency overlaps that work
        constexpr int kBv = 4;  // B float4 per thread: BN / 16 <= 4 (BN <= 64 in fp32 mode)
        auto pix_of = [&](int kb, int& n, int& oh, int& ow) {
          const int pix = kb * KP + pc;
          const bool okp = kb < kb1 && pix < p.n_pix;
          n = oh = ow = 0;
          if (okp) {
            n = static_cast<int>(fdiv(static_cast<uint32_t>(pix), p.div_OHOW));
            const int rem = pix - n * p.OH * p.OW;
            oh = static_cast<int>(fdiv(static_cast<uint32_t>(rem), p.div_OW));
            ow = rem - oh * p.OW;
          }
          return okp;
        };
        auto load_a = [&](int kb, float4 (&a)[8]) {
          int n, oh, ow;
          const bool okp = pix_of(kb, n, oh, ow);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int ih = oh * p.S + dhs[i], iw = ow * p.S + dws[i];
            const bool ok = okp && oks[i] && static_cast<unsigned>(ih) < static_cast<unsigned>(p.H) &&
                            static_cast<unsigned>(iw) < static_cast<unsigned>(p.W);
            a[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (ok)
              a[i] = __ldg(reinterpret_cast<const float4*>(
                  xs + ((static_cast<size_t>(n * p.H + ih) * p.W + iw) * p.Cs + cs[i]) * 4));
          }
        };
        float4 av[8];
        load_a(kb0, av);
        for (int kb = kb0; kb < kb1; ++kb) {
          float4 an[8], bv[kBv];
          load_a(kb + 1, an);  // past kb1: zeros, no memory access
          {
            const int pix = kb * KP + pc;
            const bool okp = pix < p.n_pix;
#pragma unroll
            for (int j = 0; j < kBv; ++j) {
              const int oc = n_tile * BN + 4 * (g0 + 4 * j);
              bv[j] = make_float4(0.f, 0.f, 0.f, 0.f);
              if (okp && 4 * (g0 + 4 * j) < BN && oc < p.OCp)
                bv[j] = __ldg(reinterpret_cast<const float4*>(p.dc32 + static_cast<size_t>(pix) * p.OCp + oc));
            }
          }
          if (!__all_sync(0xffffffffu, wait(&empty[s], par ^ 1, p.err, kSiteEmpty))) {  // warp-uniform
            alive = false;
            break;
          }
          const uint32_t a0 = sbase + s * stage_bytes;
          const uint32_t b0 = a0 + 2 * a_bytes;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rb = 4 * (g0 + 4 * i);
            const float vv[4] = {av[i].x, av[i].y, av[i].z, av[i].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int rr = rb + e;
              const uint32_t addr = a0 + rr * 128 + ((((pc >> 2) ^ (rr & 7)) << 4)) + colsw;
              uint32_t hi, lo;
              split_tf32(vv[e], hi, lo);
              st_shared_b32(addr, hi);
              st_shared_b32(addr + a_bytes, lo);
            }
          }
#pragma unroll
          for (int j = 0; j < kBv; ++j) {
            const int gb = g0 + 4 * j;
            if (4 * gb >= BN) break;  // uniform across the warp
            const float vv[4] = {bv[j].x, bv[j].y, bv[j].z, bv[j].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int rr = 4 * gb + e;
              const uint32_t addr = b0 + rr * 128 + ((((pc >> 2) ^ (rr & 7)) << 4)) + colsw;
              uint32_t hi, lo;
              split_tf32(vv[e], hi, lo);
              st_shared_b32(addr, hi);
              st_shared_b32(addr + b_bytes, lo);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&full[s]);
          if (++s == S) {
            s = 0;
            par ^= 1;
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) av[i] = an[i];
        }
      }
    }
  } else {
    // ------------------------------------------------ epilogue: partial[split][oc][k]
    const int q = warp & 3;
    const int row = q * 32 + lane;
    int tc = 0;
    for (int u = cid; u < p.num_units; u += ncl, ++tc) {
      int m_tile, n_tile, kb0, kb1;
      decode(u, m_tile, n_tile, kb0, kb1);
      const int split = u / (p.m_tiles * p.n_tiles);
      const int buf = tc & 1;
      // lane 0 waits, the warp follows: the tcgen05.ld below is warp-aligned, so
      // control flow must stay uniform even when the wait gives up
      int ok = 1;
      if (lane == 0) ok = wait(&tfull[buf], (tc >> 1) & 1, p.err, kSiteTFull) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      tc_fence_after();
      const int m = m_tile * kBM + row;
      const bool zero = kb1 <= kb0;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * acols;
      auto put = [&](int cc, const uint32_t (&r)[32]) {
        if (m >= p.Mk) return;
        float* dst = p.partial + (static_cast<size_t>(split) * p.N + n_tile * BN + cc) * p.Mk + m;
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (n_tile * BN + cc + e < p.N) dst[static_cast<size_t>(e) * p.Mk] = zero ? 0.f : __uint_as_float(r[e]);
      };
      if (ts) {  // column c holds hi x hi + lo x hi, column BN + c hi x lo
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t ra[32], rb[32];
          tmem_ld32(taddr + c0, ra);
          tmem_ld32(taddr + BN + c0, rb);
          tmem_ld_wait2(ra, rb);
#pragma unroll
          for (int e = 0; e < 32; ++e) ra[e] = __float_as_uint(__uint_as_float(ra[e]) + __uint_as_float(rb[e]));
          put(c0, ra);
        }
      } else {
        for (int c0 = 0; c0 < BN; c0 += 64) {
          uint32_t ra[32], rb[32];
          const int c1 = c0 + 32 < BN ? c0 + 32 : c0;
          tmem_ld32(taddr + c0, ra);
          tmem_ld32(taddr + c1, rb);
          tmem_ld_wait2(ra, rb);
          put(c0, ra);
          if (c0 + 32 < BN) put(c0 + 32, rb);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (pair && !leader) mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[buf]), 0));
        else mbar_arrive(&tempty[buf]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (pair) cluster_sync();  // no remote arrival or MMA write into this CTA is still in flight
  if (warp == 1) {
    tc_fence_after();
    if (pair) tmem_dealloc_pair(tmem_base, tcols);
    else tmem_dealloc(tmem_base, tcols);
  }
}

}  // namespace c2d
