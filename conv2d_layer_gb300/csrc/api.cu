// api.cu - the C ABI (include/conv2d.h): validation, workspace plan, tensor
// maps, and the launch sequence of each call.
//
// Call sequences (kernels of this library only; nothing runs on the host):
//   conv2d_fwd_train: [pack x/w] -> fprop GEMM (epilogue: + bias; no norm:
//                     also y = act; BN: per-tile statistics) -> [BN:
//                     finalize -> apply]
//   conv2d_fwd_infer: [fold BN into scale/shift] -> fprop GEMM (epilogue:
//                     y = act(acc*scale + shift))
//   conv2d_bwd:       [BN: reduce -> finalize] -> d_conv (+ dbias partials)
//                     -> finalize -> [dgrad weights -> dgrad GEMM]
//                     -> [wgrad GEMM -> split reduce]
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>

#include "conv2d.h"
#include "kernels.h"

using namespace c2d;

namespace {

// Device-side error word: kernels record the first bounded wait that ran out.
__device__ int g_error_word;

constexpr int kMaxDevices = 64;
constexpr size_t kMaxDynSmem = 232448;  // 227 KB opt-in per block

struct DevInfo {
  bool init = false;
  int sms = 0;
  int* err = nullptr;
};
std::mutex g_mu;
DevInfo g_dev[kMaxDevices];

int device_info(DevInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CONV2D_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CONV2D_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo& d = g_dev[dev];
  if (!d.init) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return CONV2D_ERR_CUDA;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err), g_error_word) != cudaSuccess) return CONV2D_ERR_CUDA;
    d.init = true;
  }
  *out = &d;
  return CONV2D_OK;
}

// SM count used for sizing when no device is visible (workspace queries on a
// machine without a GPU).
int sms_for_sizing() {
  DevInfo* d = nullptr;
  if (device_info(&d) == CONV2D_OK) return d->sms;
  cudaGetLastError();
  return 152;
}

// ------------------------------------------------------------ profiling ring
constexpr int kProfCap = 256;
struct ProfRec {
  const char* name;
  cudaEvent_t a, b;
  bool used;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
ProfRec g_prof[kProfCap];
int g_prof_head = 0, g_prof_count = 0;
bool g_prof_events = false;

int prof_begin(const char* name, cudaStream_t st) {
  if (!g_prof_on) return -1;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof_events) {
    for (int i = 0; i < kProfCap; ++i) {
      cudaEventCreate(&g_prof[i].a);
      cudaEventCreate(&g_prof[i].b);
      g_prof[i].used = false;
    }
    g_prof_events = true;
  }
  const int slot = (g_prof_head + g_prof_count) % kProfCap;
  if (g_prof_count < kProfCap)
    ++g_prof_count;
  else
    g_prof_head = (g_prof_head + 1) % kProfCap;
  g_prof[slot].name = name;
  g_prof[slot].used = true;
  cudaEventRecord(g_prof[slot].a, st);
  return slot;
}
void prof_end(int slot, cudaStream_t st) {
  if (slot < 0) return;
  cudaEventRecord(g_prof[slot].b, st);
}

#define LAUNCH(name, st, call)                \
  do {                                        \
    const int _slot = prof_begin(name, st);   \
    const cudaError_t _e = (call);            \
    prof_end(_slot, st);                      \
    if (_e != cudaSuccess) return CONV2D_ERR_CUDA; \
  } while (0)

// ------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D row-major tensor [rows][cols], 128-byte swizzled boxes of
// box_cols x box_rows; out-of-range elements read as zero.
bool encode_2d(CUtensorMap* m, const void* base, bool bf16, uint64_t cols, uint64_t rows, uint32_t box_cols,
               uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const uint64_t es = bf16 ? 2 : 4;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * es};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 weights W [OC][taps][IC] (IC a multiple of 64) as the dgrad's MN-major B operand (ConvGemmParams::
// b_mn): a 4-D view {64 input channels, OC, IC / 64 channel groups, taps}, boxes of 64 x 64 x groups x 1,
// so that one copy lands `groups` panels of 64 output-channel rows x 64 input channels of one tap.
bool encode_w_mn(CUtensorMap* m, const void* w, uint64_t OC, uint64_t taps, uint64_t IC, uint32_t groups) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || IC % 64 != 0) return false;
  cuuint64_t dims[4] = {64, OC, IC / 64, taps};
  cuuint64_t strides[3] = {taps * IC * 2, 128, IC * 2};
  cuuint32_t box[4] = {64, 64, groups, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(w), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A bf16 matrix [rows][C] (C a multiple of 64) seen as 64-channel panels: a 3-D view {64 channels, rows,
// C / 64 groups} with 128-byte swizzled boxes of 64 x box_rows x groups, so that one copy lands `groups`
// panels of box_rows rows, panel after panel (groups past C / 64 read as zeros).
bool encode_panels(CUtensorMap* m, const void* base, uint64_t C, uint64_t rows, uint32_t box_rows, uint32_t groups) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || C % 64 != 0) return false;
  cuuint64_t dims[3] = {64, rows, C / 64};
  cuuint64_t strides[2] = {C * 2, 128};
  cuuint32_t box[3] = {64, box_rows, groups};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 GEMM B operand: the tf32 hi and lo matrices [rows][cols] (hi at `hi`, lo `lo`, 16-byte aligned,
// lo after hi) seen as a 3-D tensor {cols, rows, 2 planes} whose plane stride is their distance, with
// 128-byte swizzled boxes of 32 x box_rows x 2: one copy brings a k-block's hi rows and then its lo rows.
bool encode_b_fp32(CUtensorMap* m, const void* hi, const void* lo, uint64_t cols, uint64_t rows, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const auto d = reinterpret_cast<uintptr_t>(lo) - reinterpret_cast<uintptr_t>(hi);
  if (reinterpret_cast<uintptr_t>(lo) <= reinterpret_cast<uintptr_t>(hi) || d % 16 != 0 || d < rows * cols * 4)
    return false;
  cuuint64_t dims[3] = {cols, rows, 2};
  cuuint64_t strides[2] = {cols * 4, static_cast<cuuint64_t>(d)};
  cuuint32_t box[3] = {32, box_rows, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(hi), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// B operand of the fprop / dgrad GEMM (see ConvGemmParams::tmap_b).
bool encode_b(CUtensorMap* m, bool bf, const void* hi, const void* lo, uint64_t cols, uint64_t rows,
              uint32_t box_rows) {
  return bf ? encode_2d(m, hi, true, cols, rows, 64, box_rows) : encode_b_fp32(m, hi, lo, cols, rows, box_rows);
}

typedef CUresult (*EncodeIm2colFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const int*, const int*, cuuint32_t, cuuint32_t,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeIm2colFn encode_im2col_fn() {
  static EncodeIm2colFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeIm2colFn>(p);
  });
  return fn;
}

// bf16 NHWC tensor [N][H][W][C] read by im2col TMA: boxes of `pixels` window
// corners x 64 channels, 128-byte swizzle. The corner of output (y, x) is
// (y*stride + lo_h, x*stride + lo_w); `up_h`, `up_w` place the last corner at
// (H-1+up_h, W-1+up_w). Returns false when a corner offset is outside the
// [-128, 127] range the 4-D form supports, or encoding fails.
// im2col map of an NHWC tensor of dtype dt: one 128-byte channel chunk (64 bf16 / 32 fp32) x `pixels`
// rows per copy, 128-byte swizzle. pix (elements from one pixel to the next, default C) smaller than C
// gives the folded view: "channel" c' of pixel w is element c' of the run starting at pixel w, i.e.
// channel c' % pix of pixel w + c' / pix.
bool encode_im2col(CUtensorMap* m, const void* base, int N, int H, int W, int C, int lo_h, int lo_w, int up_h,
                   int up_w, int stride, int pixels, int dt = CONV2D_BF16, int pix = 0) {
  EncodeIm2colFn fn = encode_im2col_fn();
  if (!fn) return false;
  for (int v : {lo_h, lo_w, up_h, up_w})
    if (v < -128 || v > 127) return false;
  const bool bf = dt == CONV2D_BF16;
  const cuuint64_t es = bf ? 2 : 4;
  const cuuint64_t P = pix > 0 ? static_cast<cuuint64_t>(pix) : static_cast<cuuint64_t>(C);
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(C), static_cast<cuuint64_t>(W), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(N)};
  cuuint64_t strides[3] = {P * es, static_cast<cuuint64_t>(W) * P * es, static_cast<cuuint64_t>(H) * W * P * es};
  int lower[2] = {lo_w, lo_h};
  int upper[2] = {up_w, up_h};
  cuuint32_t estr[4] = {1, static_cast<cuuint32_t>(stride), static_cast<cuuint32_t>(stride), 1};
  return fn(m, bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base),
            dims, strides, lower, upper, bf ? 64 : 32, static_cast<cuuint32_t>(pixels), estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------ geometry
long ceil_div(long a, long b) { return (a + b - 1) / b; }
long round_up(long a, long b) { return ceil_div(a, b) * b; }

struct Geo {
  int N, H, W, IC, OC, KH, KW, S, P, norm, act, dt, bn_eval, groups;
  float eps, mom;
  int OH, OW;
  long n_pix;
  int ES, EC, BKE;
  int ICp, OCp, taps;
  long Kf;
  bool pack_x;
};

int make_geo(const conv2d_desc* d, Geo* g) {
  if (!d) return CONV2D_ERR_INVALID_ARG;
  if (d->N < 1 || d->H < 1 || d->W < 1 || d->IC < 1 || d->OC < 1 || d->KH < 1 || d->KW < 1 || d->stride < 1 ||
      d->pad < 0)
    return CONV2D_ERR_INVALID_ARG;
  if (static_cast<long>(d->H) + 2L * d->pad < d->KH || static_cast<long>(d->W) + 2L * d->pad < d->KW)
    return CONV2D_ERR_INVALID_ARG;
  if (d->norm < 0 || d->norm > 3 || d->act < 0 || d->act > 3 || d->dtype < 0 || d->dtype > 1)
    return CONV2D_ERR_INVALID_ARG;
  if (d->norm != CONV2D_NORM_NONE && (!(d->eps > 0.f) || !std::isfinite(d->eps))) return CONV2D_ERR_INVALID_ARG;
  if (d->norm == CONV2D_NORM_BATCH && !(d->momentum >= 0.f && d->momentum <= 1.f)) return CONV2D_ERR_INVALID_ARG;
  if (d->norm == CONV2D_NORM_GROUP && (d->groups < 1 || d->OC % d->groups != 0)) return CONV2D_ERR_INVALID_ARG;
  if (d->stride > 8) return CONV2D_ERR_UNSUPPORTED;
  Geo& G = *g;
  G.N = d->N; G.H = d->H; G.W = d->W; G.IC = d->IC; G.OC = d->OC; G.KH = d->KH; G.KW = d->KW;
  G.S = d->stride; G.P = d->pad; G.norm = d->norm; G.act = d->act; G.dt = d->dtype;
  G.eps = d->eps; G.mom = d->momentum;
  G.bn_eval = (d->norm == CONV2D_NORM_BATCH && d->bn_eval != 0) ? 1 : 0;
  // layer norm is group norm with one group; the saved statistics have N * groups entries
  G.groups = d->norm == CONV2D_NORM_GROUP ? d->groups : 1;
  G.OH = (G.H + 2 * G.P - G.KH) / G.S + 1;
  G.OW = (G.W + 2 * G.P - G.KW) / G.S + 1;
  G.n_pix = static_cast<long>(G.N) * G.OH * G.OW;
  G.ES = G.dt == CONV2D_BF16 ? 2 : 4;
  G.EC = 16 / G.ES;
  G.BKE = 128 / G.ES;
  G.ICp = static_cast<int>(round_up(G.IC, G.EC));
  G.OCp = G.dt == CONV2D_BF16 ? (G.OC < 64 ? 64 : static_cast<int>(round_up(G.OC, 8)))
                              : static_cast<int>(round_up(G.OC, 4));
  G.taps = G.KH * G.KW;
  G.Kf = static_cast<long>(G.taps) * G.ICp;
  G.pack_x = G.ICp != G.IC;
  const long lim = INT_MAX;
  if (static_cast<long>(G.N) * G.H * G.W > lim / 2 || G.n_pix > lim / 2 || G.Kf > lim / 2 ||
      static_cast<long>(G.N) * G.H * G.W * G.ICp > (1L << 40) || G.n_pix * G.OCp > (1L << 40) ||
      static_cast<long>(G.OC) * G.Kf > lim / 2 || G.OC > 65535)
    return CONV2D_ERR_UNSUPPORTED;
  return CONV2D_OK;
}

// ------------------------------------------------------------ GEMM planning
struct Tile {
  int BN, n_tiles, stages, kps;
  size_t smem;
};

// k-blocks per shared-memory stage (ConvGemmParams::kps): with the A operand by TMA, two when at least
// three such stages fit, so that the producer, split and MMA warps pass one barrier per two k-blocks.
constexpr int kKpsMax = kMaxKps;

// Stages of `sub` bytes per k-block beside `reserve` bytes of epilogue scratch; grouped: the A operand
// comes by TMA (k-blocks may be grouped per stage).
void fit_stages(Tile& t, size_t sub, size_t reserve, bool grouped) {
  const size_t room = kMaxDynSmem - 2048 - reserve;
  t.kps = (grouped && kKpsMax > 1 && room / (kKpsMax * sub) >= 3) ? kKpsMax : 1;
  t.stages = static_cast<int>(std::min<size_t>(kMaxStages, room / (t.kps * sub)));
  t.smem = t.stages * t.kps * sub + 1024 + 512 + reserve;  // alignment slack, barriers + TMEM slot, scratch
}

// Shared-memory bytes of one k-block of a stage of the fprop / dgrad GEMM (pair: half of B per CTA).
size_t conv_sub_bytes(const Geo& g, int BN, bool ts, bool pair) {
  if (g.dt == CONV2D_BF16) return kBM * 128 + static_cast<size_t>(pair ? BN / 2 : BN) * 128;
  return (ts ? 1 : 2) * static_cast<size_t>(kBM) * 128 + 2 * static_cast<size_t>(BN) * 128;
}

// fp32 (3xTF32): the tensor core's fp32 accumulation loses a little on every MMA step (12 per k-block),
// and the loss grows with the steps that feed one accumulator, so a deep K loop accumulates in chunks of
// at most kFp32ChunkKb k-blocks (768 elements), each in its own TMEM columns, summed by the epilogue.
constexpr int kFp32ChunkKb = 24;

int fp32_chunks(long kdepth) { return static_cast<int>(std::max<long>(1, ceil_div(ceil_div(kdepth, 32), kFp32ChunkKb))); }

// kdepth: the longest K loop of a tile (elements); it bounds the column tile of fp32 GEMMs so that
// its accumulator chunks fit the 512 TMEM columns.
Tile conv_tile(const Geo& g, int ncols, long kdepth) {
  Tile t;
  int bn_max = g.dt == CONV2D_BF16 ? 256 : 128;
  if (g.dt != CONV2D_BF16) bn_max = std::max(32, std::min(bn_max, 512 / fp32_chunks(kdepth) / 32 * 32));
  t.n_tiles = static_cast<int>(ceil_div(ncols, bn_max));
  t.BN = static_cast<int>(round_up(ceil_div(ncols, t.n_tiles), 32));  // the epilogue reads 32 columns at a time
  // epilogue statistics scratch + column constants; one k-block per stage until the A path is known
  fit_stages(t, conv_sub_bytes(g, t.BN, false, false), 12 * static_cast<size_t>(t.BN) * 4, false);
  return t;
}

// fp32 GEMMs with the A operand by TMA hold A in TMEM (ConvGemmParams::ts): kTaKb * 64 TMEM columns for
// A and at least two accumulators of 2 * BN columns per chunk beside them, so BN * chunks <= 64. A stage
// then holds the raw A tiles and B's hi and lo rows. Returns false when the K loop needs more chunks.
bool ts_tile(const Geo& g, int ncols, long kdepth, Tile* out) {
  if (g.dt == CONV2D_BF16) return false;
  const int nch = fp32_chunks(kdepth);
  if (nch > 2) return false;
  Tile t;
  t.n_tiles = static_cast<int>(ceil_div(ncols, 64 / nch));
  t.BN = static_cast<int>(round_up(ceil_div(ncols, t.n_tiles), 32));
  if (t.BN * nch > 64) return false;
  fit_stages(t, conv_sub_bytes(g, t.BN, true, false), 12 * static_cast<size_t>(t.BN) * 4, true);
  *out = t;
  return true;
}

// fprop A operand by TMA im2col: whole 128-byte channel chunks, or the folded view (see fold_kw)
bool fold_kw(const Geo& g);
bool fprop_a_tma(const Geo& g) { return g.ICp % g.BKE == 0 || fold_kw(g); }

// Column tiles of the fprop GEMM (the layer-norm row partials are laid out per column tile).
int fprop_n_tiles(const Geo& g) {
  Tile t;
  if (fprop_a_tma(g) && ts_tile(g, g.OC, g.Kf, &t)) return t.n_tiles;
  return conv_tile(g, g.OC, g.Kf).n_tiles;
}

// Accumulator chunks of an fp32 GEMM whose longest tile K loop has max_kb k-blocks (see kFp32ChunkKb).
void set_chunks(ConvGemmParams& p, const Geo& g, int BN, int max_kb) {
  p.nch = 1;
  p.kpc = std::max(max_kb, 1);
  if (g.dt == CONV2D_BF16) return;
  p.nch = std::min(fp32_chunks(static_cast<long>(max_kb) * 32), 512 / BN);
  p.kpc = static_cast<int>(ceil_div(std::max(max_kb, 1), p.nch));
  p.nch = static_cast<int>(ceil_div(std::max(max_kb, 1), p.kpc));
}

// CTA pairs (cta_group::2, clusters of two) for the bf16 fprop / dgrad GEMMs whose A operand comes by
// TMA: each CTA holds half of B's columns, so a stage is smaller (more stages), and the shared-memory and
// TMA traffic per tile drops by a third. A pair's two m-tiles belong to one stride phase, so every phase
// needs an even m-tile count (every tile of a pair then holds rows of the layer). Single-phase GEMMs
// only: on the stride-2 dgrad of a 256-channel 3 x 3 layer (four phases of 4, 2, 2 and 1 taps) pairs
// measured slower (0.078 -> 0.082 ms).
constexpr bool kUsePair = true;

bool try_pair(ConvGemmParams& p, Tile& t, const Geo& g, const DevInfo* dev, const void* bmat, uint64_t bcols,
              uint64_t brows, int* grid) {
  if (!kUsePair || g.dt != CONV2D_BF16 || !p.a_tma || t.BN % 32 != 0 || p.num_phases != 1) return false;
  for (int i = 0; i < p.num_phases; ++i)
    if (ceil_div(p.ph[i].rows, kBM) & 1) return false;
  Tile pt = t;
  fit_stages(pt, conv_sub_bytes(g, t.BN, false, true), 12 * static_cast<size_t>(t.BN) * 4, true);
  const size_t smem = pt.smem;
  static std::mutex mu;
  static size_t cached_smem = 0;
  static int cached_clusters = 0;
  int clusters;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (cached_smem != smem) {
      cached_clusters = conv_gemm_pair_clusters(smem);
      cached_smem = smem;
    }
    clusters = cached_clusters;
  }
  if (clusters < 1) return false;
  CUtensorMap half;
  if (p.b_mn) {
    if ((t.BN / 2) % 64 != 0 || !encode_w_mn(&half, bmat, g.OC, g.taps, g.IC, static_cast<uint32_t>(t.BN / 128)))
      return false;
  } else if (!encode_2d(&half, bmat, true, bcols, brows, g.BKE, t.BN / 2)) {
    return false;
  }
  p.tmap_b = half;
  p.pair = 1;
  int unit = 0;  // units: pairs of m-tiles, phase by phase
  for (int i = 0; i < p.num_phases; ++i) {
    p.ph[i].unit_begin = unit;
    unit += static_cast<int>(ceil_div(p.ph[i].rows, kBM) / 2) * t.n_tiles;
  }
  p.num_units = unit;
  p.stages = pt.stages;
  p.kps = pt.kps;
  t = pt;
  *grid = 2 * std::min(p.num_units, std::min(clusters, dev->sms / 2));
  return true;
}

struct WgradPlan {
  int Mk, m_tiles, BN, n_tiles, KP, kb_total, kb_per_split, splits, stages, units;
  int rstages;  // fp32 with X by TMA: raw-tile ring
  size_t smem;
};

// fp32 weight gradient with X and d_conv by TMA (raw tiles transposed by the producer warps): the
// channels come in whole 32-float chunks.
bool wgrad_raw_tma(const Geo& g);

// fp32 layers whose kernel row covers one 128-byte run of X: KW * ICp = 32 floats of KW consecutive
// pixels (a stride-4, 4-channel, 8-wide kernel). Without horizontal padding the TMA paths read each
// kernel row as one 32-channel tap of the folded view (see encode_im2col).
bool fold_kw(const Geo& g) {
  return g.dt != CONV2D_BF16 && g.P == 0 && g.KW * g.ICp == 32 && g.ICp % 32 != 0;
}

bool wgrad_raw_tma(const Geo& g) { return g.dt != CONV2D_BF16 && (g.ICp % 32 == 0 || fold_kw(g)); }

// fused: d_conv formed in the B producer (see bwd_fused); its stages hold the pre-activation and dY boxes of
// the column tile, so the tile is at most 128 columns wide (four stages of 48 KB)
WgradPlan wgrad_plan(const Geo& g, int sms, bool fused) {
  WgradPlan w;
  const bool bf = g.dt == CONV2D_BF16;
  w.Mk = static_cast<int>(g.Kf);
  w.m_tiles = static_cast<int>(ceil_div(w.Mk, kBM));
  if (bf) {
    w.n_tiles = static_cast<int>(ceil_div(g.OC, fused ? 128 : 256));
    w.BN = static_cast<int>(round_up(ceil_div(g.OC, w.n_tiles), 64));
  } else {
    // at most 64 columns: the fp32 producers keep two k-blocks of X and one of d_conv in registers
    w.n_tiles = static_cast<int>(ceil_div(g.OC, 64));
    w.BN = static_cast<int>(round_up(ceil_div(g.OC, w.n_tiles), 32));
  }
  w.KP = bf ? 64 : 32;
  w.kb_total = static_cast<int>(ceil_div(g.n_pix, w.KP));
  const int base = w.m_tiles * w.n_tiles;
  // time model: per-CTA serial k-blocks (waves x k-blocks per split) plus the
  // HBM traffic of writing and re-reading the fp32 partials
  const double flops_kb = 2.0 * kBM * w.BN * w.KP * (bf ? 1.0 : 6.0);
  const double t_kb = flops_kb / (2.25e15 / 152.0);
  const double t_split = static_cast<double>(base) * kBM * w.BN * 8.0 / 6.8e12;
  // 3xTF32: the tensor core's fp32 accumulation is not round-to-nearest, and its error grows with the
  // number of accumulations into one TMEM accumulator; a split holds at most 32 k-blocks (1024 pixels),
  // and the splits are summed in fp64. The search starts there, so that the wave balance is chosen among
  // the allowed counts.
  const int smin = bf ? 1 : static_cast<int>(ceil_div(w.kb_total, 32));
  int best = smin;
  double best_t = 1e30;
  const int smax = std::max(smin, std::min(w.kb_total, 16 * sms));
  for (int s = smin; s <= smax; ++s) {
    const int kbp = static_cast<int>(ceil_div(w.kb_total, s));
    const int s_eff = static_cast<int>(ceil_div(w.kb_total, kbp));
    if (s_eff != s) continue;
    const long units = static_cast<long>(base) * s;
    const long waves = ceil_div(units, sms);
    const double t = waves * kbp * t_kb + s * t_split;
    if (t < best_t) {
      best_t = t;
      best = s;
    }
  }
  w.splits = best;
  w.kb_per_split = static_cast<int>(ceil_div(w.kb_total, w.splits));
  w.splits = static_cast<int>(ceil_div(w.kb_total, w.kb_per_split));
  w.units = base * w.splits;
  const size_t ns = bf ? 1 : 2;
  const size_t stage = fused ? kBM * 128 + 2 * static_cast<size_t>(w.BN) * 128
                             : ns * (kBM * 128 + static_cast<size_t>(w.BN) * 128);
  w.rstages = 0;
  if (wgrad_raw_tma(g)) {
    // A (X) in TMEM: a stage holds the d_conv hi and lo rows, and each stage has a TMEM stage of A
    // (64 columns) beside the two accumulators of 2 * BN columns; the rest of shared memory holds raw
    // tiles in flight
    // (raw stages of two k-blocks, whose copies are twice as tall, measured slower: fewer stages in flight)
    const size_t tstage = 2 * static_cast<size_t>(w.BN) * 128;
    const size_t raw = kBM * 128 + static_cast<size_t>(w.BN) * 128;
    w.stages = std::min(kMaxStages, (512 - 4 * w.BN) / 64);
    w.rstages = static_cast<int>(std::min<size_t>(kMaxStages, (kMaxDynSmem - 2048 - w.stages * tstage) / raw));
    w.smem = w.stages * tstage + w.rstages * raw + 1024 + 512;
    return w;
  }
  w.stages = static_cast<int>(std::min<size_t>(kMaxStages, (kMaxDynSmem - 2048) / stage));
  w.smem = w.stages * stage + 1024 + 512;  // alignment slack; barriers and the TMEM slot
  return w;
}

struct DgradPlan {
  int num_phases;
  ConvPhase ph[kMaxPhases];
  DgradWeightTable table;
  int Kd;
  int units;
  Tile tile;
  int ts;  // fp32 with d_conv by TMA: A in TMEM (see ts_tile)
};

// dgrad through TMA im2col: stride 1 or 2 (one map per stride phase), whole 128-byte channel chunks of
// d_conv (64 bf16 / 32 fp32).
bool dgrad_tma(const Geo& g) { return g.S * g.S <= kMaxTmaPhases && g.OCp % g.BKE == 0; }

DgradPlan dgrad_plan(const Geo& g) {
  DgradPlan d;
  std::memset(&d, 0, sizeof(d));
  d.tile = conv_tile(g, g.IC, static_cast<long>(g.taps) * g.OCp);
  d.table.flip = dgrad_tma(g) ? 1 : 0;
  d.ts = d.table.flip && ts_tile(g, g.IC, static_cast<long>(g.taps) * g.OCp, &d.tile) ? 1 : 0;
  const int S = g.S;
  int unit = 0, col = 0, n = 0;
  for (int ph_h = 0; ph_h < S; ++ph_h)
    for (int ph_w = 0; ph_w < S; ++ph_w) {
      const int Ha = ph_h < g.H ? static_cast<int>(ceil_div(g.H - ph_h, S)) : 0;
      const int Wa = ph_w < g.W ? static_cast<int>(ceil_div(g.W - ph_w, S)) : 0;
      if (Ha == 0 || Wa == 0) continue;
      const int rh = (ph_h + g.P) % S, rw = (ph_w + g.P) % S;
      const int Th = rh < g.KH ? static_cast<int>(ceil_div(g.KH - rh, S)) : 0;
      const int Tw = rw < g.KW ? static_cast<int>(ceil_div(g.KW - rw, S)) : 0;
      ConvPhase& p = d.ph[d.num_phases++];
      p.rows = g.N * Ha * Wa;
      p.Ha = Ha;
      p.Wa = Wa;
      p.qh = (ph_h + g.P - rh) / S;
      p.qw = (ph_w + g.P - rw) / S;
      p.Tw = std::max(Tw, 1);
      p.K = Th * Tw * g.OCp;
      p.num_kb = static_cast<int>(ceil_div(p.K, g.BKE));
      p.unit_begin = unit;
      p.b_col = col;
      p.oh0 = ph_h;
      p.ow0 = ph_w;
      p.Th = Th;
      p.rh = rh;
      p.rw = rw;
      p.div_Wa = make_fastdiv(Wa);
      p.div_HaWa = make_fastdiv(Ha * Wa);
      p.div_Tw = make_fastdiv(p.Tw);
      if (Th * Tw > 0) {
        d.table.col_off[n] = col;
        d.table.Th[n] = Th;
        d.table.Tw[n] = Tw;
        d.table.rh[n] = rh;
        d.table.rw[n] = rw;
        ++n;
        col += p.K;
      }
      unit += static_cast<int>(ceil_div(p.rows, kBM)) * d.tile.n_tiles;
    }
  d.table.n = n;
  d.Kd = std::max(col, g.BKE);
  d.units = unit;
  return d;
}

// dgrad with every stride phase among the columns (ConvGemmParams::seg): when KH and KW are multiples of
// the stride and so is the padding, every phase of the input grid sees the same Th x Tw taps (Th = KH / S,
// Tw = KW / S) of the same d_conv neighbourhood, so one GEMM over the coarse grid of ceil(H / S) x
// ceil(W / S) rows per image, with the S * S * IC phase-and-channel values of each S x S block of dX as its
// columns, writes dX in place: no column tile of IC columns per phase, no column buffer. Each run of
// S * IC columns is contiguous in dX (IC needs no padding), and the runs must tile the epilogue's
// 32-column chunks; d_conv comes by TMA.
bool dgrad_merged(const Geo& g) {
  if (g.S < 2 || g.KH % g.S != 0 || g.KW % g.S != 0 || g.P % g.S != 0 || g.ICp != g.IC) return false;
  return 32 % (g.S * g.IC) == 0 && g.OCp % g.BKE == 0;
}

// dgrad in column form (a 1x1 GEMM d_conv x W^T into dcol[pix][(tap, icp)], then a per-element gather)
// for strided layers with few input channels: there the stride-phase GEMMs have a column tile of IC
// padded to 32 and only KH*KW/S^2 taps each, so most of their tensor-core and operand traffic is waste.
bool dgrad_col2im(const Geo& g) {
  const size_t dcol = static_cast<size_t>(g.n_pix) * g.taps * g.ICp * g.ES;
  return g.S > 1 && g.IC <= 16 && g.OCp >= g.BKE && dcol <= (size_t(1) << 31);
}

// Batch-norm backward with d_conv formed inside the dgrad and wgrad producers, never stored: for a 1x1,
// stride-1 layer without padding d_conv is the dgrad's A operand and the wgrad's B operand as it is (each
// element read once per GEMM and column tile), so both GEMMs can read the pre-activation and dY tiles in its
// place and form it on chip (dconv_row into tensor memory for the dgrad, dconv_xform in shared memory for
// the wgrad). bf16 with whole 64-channel boxes (OC and IC multiples of 64: X by TMA in the wgrad), tanh or
// sigmoid, a streamed backward reduce (its third partial, sum (x - mean), gives dbias), and a dgrad whose
// weights stay resident in shared memory beside four 32 KB stages (at most 96 KB) as one column tile that
// leaves two TMEM accumulators beside the A stages (IC <= 192).
bool bwd_fused(const Geo& g, const RowWalk& w3) {
  return g.dt == CONV2D_BF16 && g.norm == CONV2D_NORM_BATCH && !g.bn_eval && g.KH == 1 && g.KW == 1 && g.S == 1 &&
         g.P == 0 && g.OC % 64 == 0 && g.IC % 64 == 0 && g.IC <= 192 &&
         static_cast<long>(g.OC) * g.IC * 2 <= 96 * 1024 &&
         (g.act == CONV2D_ACT_TANH || g.act == CONV2D_ACT_SIGMOID) && w3.stream && w3.cpg == 0;
}

// ------------------------------------------------------------ workspace plan
enum Reg { R_XP, R_WB, R_WBLO, R_PART, R_FOLD, R_DC, R_C12, R_WD, R_WDLO, R_WPART, R_COL, R_NREG };

struct Plan {
  size_t off[R_NREG];
  size_t total;
  RowWalk walk;
  RowWalk walk3;  // batch-norm backward reduce: three blocks per SM (its own partials and finalize)
  WgradPlan wg;
  bool fused;     // backward with d_conv formed in the GEMM producers (bwd_fused)
};

void plan_ws(const Geo& g, int op, int sms, Plan* pl) {
  size_t sz[R_NREG] = {0};
  const size_t es = g.ES;
  pl->fused = false;
  const bool ln = g.norm == CONV2D_NORM_LAYER;
  const bool gn = g.norm == CONV2D_NORM_GROUP;
  // layer and group norm walk each image as a segment of its own, statistics per group of channels
  pl->walk = make_walk(g.n_pix, g.OC, g.dt, sms, (ln || gn) ? g.N : 1, (ln || gn) ? g.OC / g.groups : 0);
  pl->walk3 = make_walk(g.n_pix, g.OC, g.dt, sms, 1, 0, 3);
  const size_t G = pl->walk.G;
  if (op == CONV2D_OP_FWD_TRAIN || op == CONV2D_OP_FWD_INFER) {
    if (g.pack_x) sz[R_XP] = static_cast<size_t>(g.N) * g.H * g.W * g.ICp * es;
    if (g.dt == CONV2D_FP32 || g.pack_x) sz[R_WB] = static_cast<size_t>(g.OC) * g.Kf * es;
    if (g.dt == CONV2D_FP32) sz[R_WBLO] = static_cast<size_t>(g.OC) * g.Kf * 4;
    if (op == CONV2D_OP_FWD_TRAIN && g.norm == CONV2D_NORM_BATCH)
      sz[R_PART] = static_cast<size_t>(ceil_div(g.n_pix, kBM)) * g.OC * 3 * 4;  // per-tile statistics
    if (ln)  // per-pixel, per-column-tile, per-half (mean, M2) of the stored conv output
      sz[R_PART] = static_cast<size_t>(g.n_pix) * std::max(conv_tile(g, g.OC, g.Kf).n_tiles, fprop_n_tiles(g)) *
                   2 * 2 * 4;
    if (gn)  // per-block, per-channel (rows, mean, M2) of the stored conv output
      sz[R_PART] = G * g.OC * 3 * 4;
    if (op == CONV2D_OP_FWD_INFER) {
      // scale, shift, then the per-(image, group) statistics of layer / group norm
      sz[R_FOLD] = (2 * static_cast<size_t>(g.OC) + 2 * static_cast<size_t>(g.N) * g.groups) * 4;
      if (ln || gn) sz[R_DC] = static_cast<size_t>(g.n_pix) * g.OC * es;  // stored conv output, normalised into y
    }
  } else {
    pl->fused = bwd_fused(g, pl->walk3);
    // the reduce with the third partial runs two blocks per SM (its registers allow no more without spills)
    if (pl->fused) pl->walk3 = make_walk(g.n_pix, g.OC, g.dt, sms, 1, 0, 2);
    if (!pl->fused) sz[R_DC] = static_cast<size_t>(g.n_pix) * g.OCp * es;
    sz[R_PART] = std::max<size_t>(G, pl->walk3.G) * g.OC * (pl->fused ? 3 : 2) * 4;
    // channel sums, then per-(image, group) sums; fused: then the per-channel terms of d_conv [4][OC]
    sz[R_C12] = 2 * (static_cast<size_t>(g.OC) + ((ln || gn) ? static_cast<size_t>(g.N) * g.groups : 0)) * 4 +
                (pl->fused ? 4 * static_cast<size_t>(g.OC) * 4 : 0);
    // dgrad weights: every phase's taps together hold each kernel tap once
    const size_t kd = std::max<size_t>(static_cast<size_t>(g.taps) * g.OCp, g.BKE);
    sz[R_WD] = static_cast<size_t>(g.ICp) * kd * es;
    if (g.dt == CONV2D_FP32) sz[R_WDLO] = static_cast<size_t>(g.ICp) * kd * 4;
    if (g.pack_x) sz[R_XP] = static_cast<size_t>(g.N) * g.H * g.W * g.ICp * es;
    if (dgrad_col2im(g) && !dgrad_merged(g)) sz[R_COL] = static_cast<size_t>(g.n_pix) * g.taps * g.ICp * es;
    pl->wg = wgrad_plan(g, sms, pl->fused);
    sz[R_WPART] = static_cast<size_t>(pl->wg.splits) * g.OC * pl->wg.Mk * 4;
  }
  size_t o = 0;
  for (int r = 0; r < R_NREG; ++r) {
    pl->off[r] = o;
    o += round_up(static_cast<long>(sz[r]), 1024);
  }
  pl->total = o;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
#define REQ_PTR(p) \
  do { if (!(p) || !aligned16(p)) return CONV2D_ERR_INVALID_ARG; } while (0)
#define OPT_PTR(p) \
  do { if ((p) && !aligned16(p)) return CONV2D_ERR_INVALID_ARG; } while (0)

char* region(void* ws, const Plan& pl, Reg r) { return static_cast<char*>(ws) + pl.off[r]; }

// fprop GEMM: D[pix][oc] = im2col(x) * B^T, epilogue per ConvGemmParams.
// stats_groups (if stats): receives the number of statistics partials written (per CTA or per tile).
// Layout of the layer-norm row partials the fprop epilogue writes: per pixel, n_tiles column tiles of BN
// columns, each in `halves` halves (two when the epilogue runs on eight warps), half 0 = hcols columns.
struct RowStatLayout {
  int n_tiles, halves, BN, hcols;
};

int run_fprop(const Geo& g, const DevInfo* dev, const void* xsrc, const void* bhi, const void* blo, void* out,
              void* out2, const float* scale, const float* shift, int out_act, float* stats, int* stats_groups,
              float* rstats, RowStatLayout* rs_layout, cudaStream_t st) {
  if (rstats && (out_act || out2)) return CONV2D_ERR_INVALID_ARG;  // row partials are of the stored value
  static ConvGemmParams p;  // guarded by g_launch_mu below (large struct)
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  std::memset(&p, 0, sizeof(p));
  Tile t = conv_tile(g, g.OC, g.Kf);
  const bool bf = g.dt == CONV2D_BF16;
  p.src = xsrc;
  p.Hs = g.H;
  p.Ws = g.W;
  p.Cs = g.ICp;
  p.rs = g.S;
  p.tap_sign = 1;
  p.div_Cs = make_fastdiv(g.ICp);
  p.num_phases = 1;
  ConvPhase& ph = p.ph[0];
  ph.rows = static_cast<int>(g.n_pix);
  ph.Ha = g.OH;
  ph.Wa = g.OW;
  ph.qh = -g.P;
  ph.qw = -g.P;
  ph.Tw = g.KW;
  ph.K = static_cast<int>(g.Kf);
  ph.num_kb = static_cast<int>(ceil_div(g.Kf, g.BKE));
  ph.unit_begin = 0;
  ph.b_col = 0;
  ph.div_Wa = make_fastdiv(g.OW);
  ph.div_HaWa = make_fastdiv(g.OH * g.OW);
  ph.div_Tw = make_fastdiv(g.KW);
  p.N = g.OC;
  p.out = out;
  p.out2 = out2;
  p.out_ld = g.OC;
  p.Ho = g.OH;
  p.Wo = g.OW;
  p.os = 1;
  p.ep_scale = scale;
  p.ep_shift = shift;
  p.act = g.act;
  p.out_act = out_act;
  p.stats = stats;
  p.rstats = rstats;
  // A by TMA im2col when the channels come in whole 128-byte chunks (64 bf16 / 32 fp32), or through the
  // folded view (one 32-float run per kernel row: the taps are the KH rows, Tw = 1)
  if (g.ICp % g.BKE == 0 &&
      encode_im2col(&p.tmap_a[0], xsrc, g.N, g.H, g.W, g.ICp, -g.P, -g.P, (g.OH - 1) * g.S - g.P - (g.H - 1),
                    (g.OW - 1) * g.S - g.P - (g.W - 1), g.S, kBM, g.dt)) {
    p.a_tma = 1;
    p.a_chunks = g.ICp / g.BKE;
    ph.a_lo_h = -g.P;
    ph.a_lo_w = -g.P;
    ph.a_map = 0;
  } else if (fold_kw(g) &&
             encode_im2col(&p.tmap_a[0], xsrc, g.N, g.H, g.W, g.KW * g.ICp, -g.P, -g.P,
                           (g.OH - 1) * g.S - g.P - (g.H - 1), (g.OW - 1) * g.S - g.P - (g.W - 1), g.S, kBM, g.dt,
                           g.ICp)) {
    p.a_tma = 1;
    p.a_chunks = 1;
    ph.Tw = 1;
    ph.div_Tw = make_fastdiv(1);
    ph.a_lo_h = -g.P;
    ph.a_lo_w = -g.P;
    ph.a_map = 0;
  }
  // fp32 with A by TMA: A in TMEM when the K loop allows it (see ts_tile); bf16 with A by TMA: k-blocks
  // grouped per stage
  if (!bf && p.a_tma && ts_tile(g, g.OC, g.Kf, &t)) p.ts = 1;
  if (bf && p.a_tma) fit_stages(t, conv_sub_bytes(g, t.BN, false, false), 12 * static_cast<size_t>(t.BN) * 4, true);
  if (!encode_b(&p.tmap_b, bf, bhi, blo, g.Kf, g.OC, t.BN)) return CONV2D_ERR_CUDA;
  p.n_tiles = t.n_tiles;
  p.BN = t.BN;
  p.num_units = static_cast<int>(ceil_div(g.n_pix, kBM)) * t.n_tiles;
  p.stages = t.stages;
  p.kps = t.kps;
  p.err = dev->err;
  set_chunks(p, g, t.BN, ph.num_kb);
  if (bf && !p.a_tma && t.stages < kLag + 1) return CONV2D_ERR_UNSUPPORTED;  // the gather's copies in flight
  if (rs_layout) {
    const bool ep8 = bf && p.a_tma;  // the kernel's eight-warp epilogue splits the columns in two halves
    rs_layout->n_tiles = t.n_tiles;
    rs_layout->halves = ep8 ? 2 : 1;
    rs_layout->BN = t.BN;
    rs_layout->hcols = ep8 ? 32 * ((t.BN / 32 + 1) / 2) : t.BN;
  }
  int grid = std::min(p.num_units, dev->sms);
  if (bf) try_pair(p, t, g, dev, bhi, g.Kf, g.OC, &grid);
  p.stats_per_cta = t.n_tiles == 1 ? 1 : 0;
  if (stats_groups) *stats_groups = p.stats_per_cta ? grid : static_cast<int>(ceil_div(g.n_pix, kBM));
  LAUNCH("fprop_gemm", st, bf ? launch_conv_gemm_bf16(p, grid, t.smem, st) : launch_conv_gemm_tf32(p, grid, t.smem, st));
  return CONV2D_OK;
}

// Column-form dgrad (see dgrad_col2im): dcol = d_conv [n_pix][OCp] x B[(tap, icp)][oc] as the fprop of a
// 1x1 convolution over the d_conv image, then dX gathered per element.
int run_dgrad_col2im(const Geo& g, const DevInfo* dev, const void* w, const void* dconv, void* dx, void* ws,
                     const Plan& pl, cudaStream_t st) {
  void* bhi = region(ws, pl, R_WD);
  float* blo = reinterpret_cast<float*>(region(ws, pl, R_WDLO));
  const bool bf = g.dt == CONV2D_BF16;
  LAUNCH("dgrad_weights", st,
         launch_prep_col2im_weights(g.dt, w, bhi, bf ? nullptr : blo, g.OC, g.taps, g.IC, g.ICp, g.OCp, st));
  conv2d_desc d2;
  std::memset(&d2, 0, sizeof(d2));
  d2.N = g.N; d2.H = g.OH; d2.W = g.OW; d2.IC = g.OCp; d2.OC = g.taps * g.ICp;
  d2.KH = 1; d2.KW = 1; d2.stride = 1; d2.pad = 0;
  d2.norm = CONV2D_NORM_NONE; d2.act = CONV2D_ACT_IDENTITY; d2.dtype = g.dt;
  Geo g2;
  int rc = make_geo(&d2, &g2);
  if (rc) return rc;
  void* dcol = region(ws, pl, R_COL);
  if ((rc = run_fprop(g2, dev, dconv, bhi, bf ? nullptr : blo, dcol, nullptr, nullptr, nullptr, 0, nullptr, nullptr,
                      nullptr, nullptr, st)))
    return rc;
  LAUNCH("dgrad_col2im", st,
         launch_col2im(g.dt, dcol, dx, g.N, g.H, g.W, g.IC, g.ICp, g.OH, g.OW, g.KH, g.KW, g.S, g.P, st));
  return CONV2D_OK;
}

// Phase-merged dgrad (see dgrad_merged): one GEMM over the coarse grid, d_conv by TMA im2col with the
// Th x Tw window, B = the merged weights, the epilogue storing each row as S runs of S * IC values.
int run_dgrad_merged(const Geo& g, const DevInfo* dev, const void* w, const void* dconv, void* dx, void* ws,
                     const Plan& pl, cudaStream_t st) {
  static ConvGemmParams p;
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  const bool bf = g.dt == CONV2D_BF16;
  const int S = g.S, Th = g.KH / S, Tw = g.KW / S, p0 = g.P / S;
  const int ncols = S * S * g.ICp;
  const int Kd = Th * Tw * g.OCp;
  void* whi = region(ws, pl, R_WD);
  float* wlo = reinterpret_cast<float*>(region(ws, pl, R_WDLO));
  LAUNCH("dgrad_weights", st,
         launch_prep_dgrad_merged_weights(g.dt, w, whi, bf ? nullptr : wlo, g.OC, g.KH, g.KW, g.IC, g.ICp, g.OCp,
                                          S, st));
  std::memset(&p, 0, sizeof(p));
  Tile t;
  p.ts = (!bf && ts_tile(g, ncols, Kd, &t)) ? 1 : 0;
  if (!p.ts) {
    t = conv_tile(g, ncols, Kd);
    if (bf) fit_stages(t, conv_sub_bytes(g, t.BN, false, false), 12 * static_cast<size_t>(t.BN) * 4, true);
  }
  if (!encode_b(&p.tmap_b, bf, whi, wlo, Kd, ncols, t.BN)) return CONV2D_ERR_CUDA;
  const int Ha = static_cast<int>(ceil_div(g.H, S)), Wa = static_cast<int>(ceil_div(g.W, S));
  p.src = dconv;
  p.Hs = g.OH;
  p.Ws = g.OW;
  p.Cs = g.OCp;
  p.rs = 1;
  p.tap_sign = -1;
  p.div_Cs = make_fastdiv(g.OCp);
  p.num_phases = 1;
  ConvPhase& ph = p.ph[0];
  ph.rows = g.N * Ha * Wa;
  ph.Ha = Ha;
  ph.Wa = Wa;
  ph.qh = p0;
  ph.qw = p0;
  ph.Tw = Tw;
  ph.K = Kd;
  ph.num_kb = static_cast<int>(ceil_div(Kd, g.BKE));
  ph.div_Wa = make_fastdiv(Wa);
  ph.div_HaWa = make_fastdiv(Ha * Wa);
  ph.div_Tw = make_fastdiv(Tw);
  // row (a, b) reads d_conv at (a + p0 - t', b + p0 - u') for the kernel taps (ph + S t', ph + S u'): with
  // the window corner (a + p0 - (Th - 1), b + p0 - (Tw - 1)) the im2col offsets are the reversed taps
  ph.a_lo_h = p0 - (Th - 1);
  ph.a_lo_w = p0 - (Tw - 1);
  if (!encode_im2col(&p.tmap_a[0], dconv, g.N, g.OH, g.OW, g.OCp, ph.a_lo_h, ph.a_lo_w,
                     (Ha - 1) + ph.a_lo_h - (g.OH - 1), (Wa - 1) + ph.a_lo_w - (g.OW - 1), 1, kBM, g.dt))
    return CONV2D_ERR_CUDA;
  p.a_tma = 1;
  p.a_chunks = g.OCp / g.BKE;
  p.n_tiles = t.n_tiles;
  p.BN = t.BN;
  p.N = ncols;
  p.num_units = static_cast<int>(ceil_div(ph.rows, kBM)) * t.n_tiles;
  p.out = dx;
  p.out_ld = g.IC;
  p.Ho = g.H;
  p.Wo = g.W;
  p.os = S;
  p.seg = S * g.IC;
  p.seg_ld = g.W * g.IC;
  while ((1 << p.seg_sh) < p.seg) ++p.seg_sh;  // powers of two (dgrad_merged)
  while ((1 << p.ic_sh) < g.IC) ++p.ic_sh;
  p.out_h = g.H;
  p.out_w = g.W;
  p.stages = t.stages;
  p.kps = t.kps;
  p.err = dev->err;
  set_chunks(p, g, t.BN, ph.num_kb);
  int grid = std::min(p.num_units, dev->sms);
  if (bf) try_pair(p, t, g, dev, whi, Kd, ncols, &grid);
  LAUNCH("dgrad_gemm", st,
         bf ? launch_conv_gemm_bf16(p, grid, t.smem, st) : launch_conv_gemm_tf32(p, grid, t.smem, st));
  return CONV2D_OK;
}

// Operands of a backward with d_conv formed in the GEMM producers (see bwd_fused): the layer's stored
// pre-activation, dY and the per-channel terms of d_conv [4][OC].
struct XfSrc {
  const void* pre;
  const void* dy;
  const float* tbl;
};

int run_dgrad(const Geo& g, const DevInfo* dev, const void* w, const void* dconv, void* dx, void* ws,
              const Plan& pl, cudaStream_t st, const XfSrc* xf = nullptr) {
  if (xf && (g.S != 1 || g.KH != 1 || g.KW != 1 || g.P != 0)) return CONV2D_ERR_INVALID_ARG;
  if (dgrad_merged(g)) return run_dgrad_merged(g, dev, w, dconv, dx, ws, pl, st);
  if (dgrad_col2im(g)) return run_dgrad_col2im(g, dev, w, dconv, dx, ws, pl, st);
  static ConvGemmParams p;
  static DgradPlan d;
  static std::mutex mu;
  std::lock_guard<std::mutex> lk(mu);
  const bool bf = g.dt == CONV2D_BF16;
  d = dgrad_plan(g);
  void* whi = region(ws, pl, R_WD);
  float* wlo = reinterpret_cast<float*>(region(ws, pl, R_WDLO));
  std::memset(&p, 0, sizeof(p));
  // bf16 with d_conv by TMA over several stride phases, whole 64-channel groups: the weights as an MN-major B
  // operand, no transposed copy (`mixed` layer 2: 0.5225 -> 0.5165 ms a step). A one-phase dgrad keeps the
  // copy: there, with CTA pairs, the strided reads of W cost what the copy saves (`large` 2.006 -> 2.009 ms).
  const bool b_mn = bf && !xf && d.table.flip && d.num_phases > 1 && g.IC % 64 == 0 && g.OC == g.OCp &&
                    d.tile.BN % 64 == 0;
  if (b_mn) {
    if (!encode_w_mn(&p.tmap_b, w, g.OC, g.taps, g.IC, static_cast<uint32_t>(d.tile.BN / 64))) return CONV2D_ERR_CUDA;
    p.b_mn = 1;
    p.S = g.S;
    p.KW = g.KW;
    whi = const_cast<void*>(w);
  } else {
    LAUNCH("dgrad_weights", st,
           launch_prep_dgrad_weights(g.dt, w, whi, bf ? nullptr : wlo, g.OC, g.KH, g.KW, g.IC, g.ICp, g.OCp, g.S, d.Kd,
                                     d.table, st));
    if (!encode_b(&p.tmap_b, bf, whi, wlo, d.Kd, g.ICp, d.tile.BN)) return CONV2D_ERR_CUDA;
  }
  p.src = dconv;
  p.Hs = g.OH;
  p.Ws = g.OW;
  p.Cs = g.OCp;
  p.rs = 1;
  p.tap_sign = -1;
  p.div_Cs = make_fastdiv(g.OCp);
  p.num_phases = d.num_phases;
  for (int i = 0; i < d.num_phases; ++i) p.ph[i] = d.ph[i];
  p.n_tiles = d.tile.n_tiles;
  p.BN = d.tile.BN;
  p.N = g.IC;
  p.num_units = d.units;
  p.out = dx;
  p.out2 = nullptr;
  p.out_ld = g.IC;
  p.Ho = g.H;
  p.Wo = g.W;
  p.os = g.S;
  p.act = 0;
  p.out_act = 0;
  if (xf) {
    // A = d_conv [n_pix][OC] formed from the pre-activation and dY tiles (ConvGemmParams::xf)
    if (!encode_2d(&p.tmap_a[0], xf->pre, true, g.OC, g.n_pix, 64, kBM) ||
        !encode_2d(&p.tmap_a[1], xf->dy, true, g.OC, g.n_pix, 64, kBM))
      return CONV2D_ERR_CUDA;
    p.a_tma = 1;
    p.a_chunks = 1;
    p.xf = 1;
    p.xf_C = g.OC;
    p.xf_tbl = xf->tbl;
    p.act = g.act;
  } else if (d.table.flip) {
    // One im2col map per stride phase. Phase row (a, b) reads d_conv at (a + qh - tt, b + qw - uu) for
    // its taps (tt, uu) < (Th, Tw): with the window corner (a + qh - (Th - 1), b + qw - (Tw - 1)) the
    // tap offsets are the flipped indices (Th - 1 - tt, Tw - 1 - uu), matching the flipped weight
    // columns, and the map walks the phase's own Ha x Wa grid.
    for (int i = 0; i < d.num_phases; ++i) {
      ConvPhase& ph = p.ph[i];
      const int Th = ph.K / (ph.Tw * g.OCp);
      ph.a_map = i;
      ph.a_lo_h = ph.qh - (Th - 1);
      ph.a_lo_w = ph.qw - (ph.Tw - 1);
      if (ph.num_kb == 0) continue;  // no taps: nothing is loaded
      if (!encode_im2col(&p.tmap_a[i], dconv, g.N, g.OH, g.OW, g.OCp, ph.a_lo_h, ph.a_lo_w,
                         (ph.Ha - 1) + ph.a_lo_h - (g.OH - 1), (ph.Wa - 1) + ph.a_lo_w - (g.OW - 1), 1, kBM, g.dt))
        return CONV2D_ERR_CUDA;
    }
    p.a_tma = 1;
    p.a_chunks = g.OCp / g.BKE;
    p.ts = d.ts;
  }
  if (p.xf) {
    // a stage: the pre-activation and dY tiles of one k-block; B resident (one column tile), then the
    // epilogue scratch and the terms of d_conv
    if (d.tile.n_tiles != 1 || d.num_phases != 1) return CONV2D_ERR_INVALID_ARG;
    p.bres = static_cast<uint32_t>(d.ph[0].num_kb * d.tile.BN * 128);
    fit_stages(d.tile, 2 * kBM * 128,
               (12 * static_cast<size_t>(d.tile.BN) + 4 * static_cast<size_t>(g.OC)) * 4 + p.bres, false);
    if (d.tile.stages < 2) return CONV2D_ERR_UNSUPPORTED;
  } else if (bf && p.a_tma) {
    fit_stages(d.tile, conv_sub_bytes(g, d.tile.BN, false, false), 12 * static_cast<size_t>(d.tile.BN) * 4, true);
  }
  p.stages = d.tile.stages;
  p.kps = d.tile.kps;
  p.err = dev->err;
  {
    int max_kb = 0;
    for (int i = 0; i < d.num_phases; ++i) max_kb = std::max(max_kb, d.ph[i].num_kb);
    set_chunks(p, g, d.tile.BN, max_kb);
  }
  if (bf && !p.a_tma && d.tile.stages < kLag + 1) return CONV2D_ERR_UNSUPPORTED;  // the gather's copies
  int grid = std::min(p.num_units, dev->sms);
  if (bf && !p.xf) try_pair(p, d.tile, g, dev, whi, d.Kd, g.ICp, &grid);
  LAUNCH("dgrad_gemm", st,
         bf ? launch_conv_gemm_bf16(p, grid, d.tile.smem, st) : launch_conv_gemm_tf32(p, grid, d.tile.smem, st));
  return CONV2D_OK;
}

// bpart, bG, dbias: the dbias partials [bG][OC] summed into dbias by the split reduce's launch (null: none).
int run_wgrad(const Geo& g, const DevInfo* dev, const void* xsrc, const void* dconv, float* dw, void* ws,
              const Plan& pl, cudaStream_t st, const XfSrc* xf = nullptr, const float* bpart = nullptr, int bG = 0,
              float* dbias = nullptr) {
  WgradParams p;
  std::memset(&p, 0, sizeof(p));
  const WgradPlan& w = pl.wg;
  const bool bf = g.dt == CONV2D_BF16;
  if (xf && (!bf || g.ICp % 64 != 0 || g.OCp != g.OC)) return CONV2D_ERR_INVALID_ARG;
  if (bf && !xf && !encode_2d(&p.tmap_dc, dconv, true, g.OCp, g.n_pix, 64, 64)) return CONV2D_ERR_CUDA;
  if (xf) {  // B = d_conv formed from the pre-activation (tmap_dc) and dY panels (WgradParams::xf)
    if (!encode_panels(&p.tmap_dc, xf->pre, g.OC, g.n_pix, 64, w.BN / 64) ||
        !encode_panels(&p.tmap_dy, xf->dy, g.OC, g.n_pix, 64, w.BN / 64))
      return CONV2D_ERR_CUDA;
    p.xf = 1;
    p.xf_C = g.OC;
    p.xf_tbl = xf->tbl;
    p.act = g.act;
  }
  p.x = xsrc;
  p.dc32 = bf ? nullptr : static_cast<const float*>(dconv);
  p.H = g.H;
  p.W = g.W;
  p.Cs = g.ICp;
  p.OH = g.OH;
  p.OW = g.OW;
  p.S = g.S;
  p.P = g.P;
  p.KW = g.KW;
  p.div_Cs = make_fastdiv(g.ICp);
  p.div_KW = make_fastdiv(g.KW);
  p.div_OW = make_fastdiv(g.OW);
  p.div_OHOW = make_fastdiv(g.OH * g.OW);
  p.Mk = w.Mk;
  p.m_tiles = w.m_tiles;
  p.n_tiles = w.n_tiles;
  p.BN = w.BN;
  p.N = g.OC;
  p.OCp = g.OCp;
  p.n_pix = static_cast<int>(g.n_pix);
  p.kb_total = w.kb_total;
  p.kb_per_split = w.kb_per_split;
  p.splits = w.splits;
  p.num_units = w.units;
  p.partial = reinterpret_cast<float*>(region(ws, pl, R_WPART));
  if (xf) {  // 1x1, stride 1: X [n_pix][ICp] as two 64-channel panels per m-tile, one copy
    if (!encode_panels(&p.tmap_x, xsrc, g.ICp, g.n_pix, 64, 2)) return CONV2D_ERR_CUDA;
    p.a_tma = 1;
  } else if (bf && g.ICp % 64 == 0 &&
             encode_im2col(&p.tmap_x, xsrc, g.N, g.H, g.W, g.ICp, -g.P, -g.P, (g.OH - 1) * g.S - g.P - (g.H - 1),
                           (g.OW - 1) * g.S - g.P - (g.W - 1), g.S, w.KP)) {
    p.a_tma = 1;
  }
  if (wgrad_raw_tma(g)) {
    // folded view: the rows of the weight gradient are (kh, kw, ic) with one 32-float run per kh, i.e.
    // 32-channel chunks of KW = 1 taps
    const bool fold = fold_kw(g);
    const int cs = fold ? g.KW * g.ICp : g.ICp;
    if (!encode_im2col(&p.tmap_x, xsrc, g.N, g.H, g.W, cs, -g.P, -g.P, (g.OH - 1) * g.S - g.P - (g.H - 1),
                       (g.OW - 1) * g.S - g.P - (g.W - 1), g.S, w.KP, g.dt, g.ICp) ||
        !encode_2d(&p.tmap_dc, dconv, false, g.OCp, g.n_pix, 32, 32))
      return CONV2D_ERR_CUDA;
    p.a_tma = 1;
    p.ts = 1;
    p.rstages = w.rstages;
    if (fold) {
      p.Cs = cs;
      p.div_Cs = make_fastdiv(cs);
      p.KW = 1;
      p.div_KW = make_fastdiv(1);
    }
  }
  p.stages = w.stages;
  p.kps = 1;
  p.err = dev->err;
  if (bf && !p.a_tma && w.stages < kLag + 1) return CONV2D_ERR_UNSUPPORTED;  // the gather's copies in flight
  int grid = std::min(p.num_units, dev->sms);
  size_t smem = w.smem;
  if (bf && p.a_tma) {  // k-blocks grouped per stage, each copy covering them all (WgradParams::kps)
    Tile t;
    if (p.xf)  // the X panels, the pre-activation and the dY boxes; one k-block per stage; the terms of d_conv
      fit_stages(t, kBM * 128 + 2 * static_cast<size_t>(w.BN) * 128, 4 * static_cast<size_t>(g.OC) * 4, false);
    else
      fit_stages(t, kBM * 128 + static_cast<size_t>(w.BN) * 128, 0, true);
    p.stages = t.stages;
    p.kps = t.kps;
    smem = t.smem;
  }
  if (p.xf && !p.a_tma) return CONV2D_ERR_UNSUPPORTED;
  // CTA pairs: two m-tiles per pair, each CTA with half of the d_conv columns
  if (kUsePair && bf && p.a_tma && !p.xf && (w.m_tiles % 2) == 0 && w.BN % 128 == 0) {
    Tile pt;
    fit_stages(pt, kBM * 128 + static_cast<size_t>(w.BN / 2) * 128, 0, true);
    const int stages = pt.stages;
    const size_t psmem = pt.smem;
    static std::mutex mu;
    static size_t cached_smem = 0;
    static int cached_clusters = 0;
    int clusters;
    {
      std::lock_guard<std::mutex> lk(mu);
      if (cached_smem != psmem) {
        cached_clusters = wgrad_gemm_pair_clusters(psmem);
        cached_smem = psmem;
      }
      clusters = cached_clusters;
    }
    if (clusters > 0) {
      p.pair = 1;
      p.m_tiles = w.m_tiles / 2;
      p.num_units = w.units / 2;
      p.stages = stages;
      p.kps = pt.kps;
      smem = psmem;
      grid = 2 * std::min(p.num_units, std::min(clusters, dev->sms / 2));
    }
  }
  if (bf && p.kps > 1) {  // copies of kps k-blocks: X panels and d_conv boxes kps * 64 pixels tall
    if (!encode_im2col(&p.tmap_x, xsrc, g.N, g.H, g.W, g.ICp, -g.P, -g.P, (g.OH - 1) * g.S - g.P - (g.H - 1),
                       (g.OW - 1) * g.S - g.P - (g.W - 1), g.S, w.KP * p.kps) ||
        !encode_2d(&p.tmap_dc, dconv, true, g.OCp, g.n_pix, 64, 64 * p.kps))
      return CONV2D_ERR_CUDA;
  }
  LAUNCH("wgrad_gemm", st,
         bf ? launch_wgrad_gemm_bf16(p, grid, smem, st) : launch_wgrad_gemm_tf32(p, grid, smem, st));
  LAUNCH("wgrad_reduce", st,
         launch_wgrad_reduce(p.partial, w.splits, g.OC, g.taps, g.ICp, g.IC, dw, bpart, bG, dbias, st));
  return CONV2D_OK;
}

// Pack x (and w) to ICp channels when IC is not a multiple of the 16-byte
// vector; for fp32 split w into tf32 hi / lo. Returns the GEMM operands.
int prep_forward_operands(const Geo& g, const void* x, const void* w, void* ws, const Plan& pl, const void** xsrc,
                          const void** bhi, const void** blo, cudaStream_t st) {
  *xsrc = x;
  *bhi = w;
  *blo = nullptr;
  if (g.pack_x) {
    void* xp = region(ws, pl, R_XP);
    LAUNCH("pack_x", st, launch_pack_channels(g.dt, x, xp, static_cast<long>(g.N) * g.H * g.W, g.IC, g.ICp, st));
    *xsrc = xp;
  }
  if (g.dt == CONV2D_FP32 || g.pack_x) {
    void* wb = region(ws, pl, R_WB);
    float* wl = reinterpret_cast<float*>(region(ws, pl, R_WBLO));
    LAUNCH("prep_w", st,
           launch_prep_fprop_weights(g.dt, w, wb, g.dt == CONV2D_FP32 ? wl : nullptr, g.OC, g.taps, g.IC, g.ICp, st));
    *bhi = wb;
    if (g.dt == CONV2D_FP32) *blo = wl;
  }
  return CONV2D_OK;
}

// One thread waits on a barrier that nothing completes: the library's bounded
// wait must give up, record `site` in the error word and let the kernel end.
__global__ void wait_limit_selftest_kernel(int* err, int site) {
  pdl_entry();
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)wait(&bar, 0, err, site);
}

}  // namespace

extern "C" {

int conv2d_selftest_wait_limit(void* stream) {
  DevInfo* dev = nullptr;
  const int rc = device_info(&dev);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  LAUNCH("wait_limit_selftest", st, (launch_k(wait_limit_selftest_kernel, 1, 32, 0, st, 1, dev->err, 6), cudaGetLastError()));
  return CONV2D_OK;
}


int conv2d_out_hw(const conv2d_desc* desc, int32_t* OH, int32_t* OW) {
  Geo g;
  const int rc = make_geo(desc, &g);
  if (rc == CONV2D_ERR_INVALID_ARG) return rc;
  if (!desc || !OH || !OW) return CONV2D_ERR_INVALID_ARG;
  *OH = (desc->H + 2 * desc->pad - desc->KH) / desc->stride + 1;
  *OW = (desc->W + 2 * desc->pad - desc->KW) / desc->stride + 1;
  return CONV2D_OK;
}

int conv2d_validate(const conv2d_desc* desc) {
  Geo g;
  return make_geo(desc, &g);
}

size_t conv2d_workspace_size(const conv2d_desc* desc, int op) {
  Geo g;
  if (make_geo(desc, &g) != CONV2D_OK) return 0;
  if (op < 0 || op > 2) return 0;
  Plan pl;
  plan_ws(g, op, sms_for_sizing(), &pl);
  return pl.total;
}

int conv2d_fwd_train(const conv2d_desc* desc, const void* x, const void* w, const float* bias, const float* gamma,
                     const float* beta, float* running_mean, float* running_var, void* pre_act, float* save_mean,
                     float* save_inv_std, void* y, void* ws, size_t ws_bytes, void* stream) {
  Geo g;
  int rc = make_geo(desc, &g);
  if (rc) return rc;
  REQ_PTR(x); REQ_PTR(w); REQ_PTR(pre_act); REQ_PTR(y); OPT_PTR(bias);
  if (g.norm == CONV2D_NORM_BATCH) {
    REQ_PTR(gamma); REQ_PTR(beta); REQ_PTR(running_mean); REQ_PTR(running_var); REQ_PTR(save_mean);
    REQ_PTR(save_inv_std);
  }
  if (g.norm == CONV2D_NORM_LAYER || g.norm == CONV2D_NORM_GROUP) {
    REQ_PTR(gamma); REQ_PTR(beta); REQ_PTR(save_mean); REQ_PTR(save_inv_std);
  }
  DevInfo* dev = nullptr;
  if ((rc = device_info(&dev))) return rc;
  Plan pl;
  plan_ws(g, CONV2D_OP_FWD_TRAIN, dev->sms, &pl);
  pl.walk.err = dev->err;
  if (!ws || ws_bytes < pl.total || (reinterpret_cast<uintptr_t>(ws) & 255u)) return CONV2D_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const void *xsrc, *bhi, *blo;
  if ((rc = prep_forward_operands(g, x, w, ws, pl, &xsrc, &bhi, &blo, st))) return rc;
  const bool bn = g.norm == CONV2D_NORM_BATCH;
  if (g.norm == CONV2D_NORM_LAYER) {
    // layer norm: per-image statistics of the stored conv output from the epilogue's row partials
    float* rs = reinterpret_cast<float*>(region(ws, pl, R_PART));
    RowStatLayout lay;
    if ((rc = run_fprop(g, dev, xsrc, bhi, blo, pre_act, nullptr, nullptr, bias, 0, nullptr, nullptr, rs, &lay,
                        st)))
      return rc;
    LAUNCH("ln_stats_finalize", st,
           launch_ln_stats_finalize(rs, g.N, static_cast<long>(g.OH) * g.OW, lay.n_tiles, lay.halves, lay.BN,
                                    lay.hcols, g.OC, g.eps, save_mean, save_inv_std, st));
    // reversed: starts on the last rows of pre_act, which the fprop epilogue wrote last
    LAUNCH("ln_apply", st,
           launch_bn_apply(g.dt, pre_act, y, pl.walk, save_mean, save_inv_std, gamma, beta, g.act, 1, st));
    return CONV2D_OK;
  }
  if (g.norm == CONV2D_NORM_GROUP) {
    // group norm: per-channel partials of the stored conv output on an image-aligned walk (reversed: it
    // starts on the rows the fprop epilogue wrote last), merged per (image, group); then the apply
    float* gp = reinterpret_cast<float*>(region(ws, pl, R_PART));
    if ((rc = run_fprop(g, dev, xsrc, bhi, blo, pre_act, nullptr, nullptr, bias, 0, nullptr, nullptr, nullptr,
                        nullptr, st)))
      return rc;
    LAUNCH("gn_stats", st, launch_norm_stats(g.dt, pre_act, pl.walk, 1, gp, st));
    LAUNCH("gn_stats_finalize", st, launch_gn_stats_finalize(gp, pl.walk, g.eps, save_mean, save_inv_std, st));
    LAUNCH("gn_apply", st,
           launch_bn_apply(g.dt, pre_act, y, pl.walk, save_mean, save_inv_std, gamma, beta, g.act, 0, st));
    return CONV2D_OK;
  }
  float* part = (bn && !g.bn_eval) ? reinterpret_cast<float*>(region(ws, pl, R_PART)) : nullptr;
  int groups = 0;
  if ((rc = run_fprop(g, dev, xsrc, bhi, blo, pre_act, bn ? nullptr : y, nullptr, bias, 0, part, &groups, nullptr,
                      nullptr, st)))
    return rc;
  if (bn && g.bn_eval) {
    // evaluation mode: normalise with the running statistics, update nothing
    LAUNCH("bn_eval_stats", st, launch_bn_eval_stats(running_mean, running_var, g.eps, g.OC, save_mean, save_inv_std, st));
    LAUNCH("bn_apply", st,
           launch_bn_apply(g.dt, pre_act, y, pl.walk, save_mean, save_inv_std, gamma, beta, g.act, 1, st));
  } else if (bn) {
    RowWalk tiles = pl.walk;  // statistics partials written by the fprop GEMM
    tiles.G = groups;
    LAUNCH("bn_stats_finalize", st,
           launch_bn_stats_finalize(part, tiles, g.eps, g.mom, save_mean, save_inv_std, running_mean, running_var,
                                    st));
    LAUNCH("bn_apply", st,
           launch_bn_apply(g.dt, pre_act, y, pl.walk, save_mean, save_inv_std, gamma, beta, g.act, 1, st));
  }
  return CONV2D_OK;
}

int conv2d_fwd_infer(const conv2d_desc* desc, const void* x, const void* w, const float* bias, const float* gamma,
                     const float* beta, const float* running_mean, const float* running_var, void* y, void* ws,
                     size_t ws_bytes, void* stream) {
  Geo g;
  int rc = make_geo(desc, &g);
  if (rc) return rc;
  REQ_PTR(x); REQ_PTR(w); REQ_PTR(y); OPT_PTR(bias);
  if (g.norm == CONV2D_NORM_BATCH) {
    REQ_PTR(gamma); REQ_PTR(beta); REQ_PTR(running_mean); REQ_PTR(running_var);
  }
  if (g.norm == CONV2D_NORM_LAYER || g.norm == CONV2D_NORM_GROUP) {
    REQ_PTR(gamma); REQ_PTR(beta);
  }
  DevInfo* dev = nullptr;
  if ((rc = device_info(&dev))) return rc;
  Plan pl;
  plan_ws(g, CONV2D_OP_FWD_INFER, dev->sms, &pl);
  pl.walk.err = dev->err;
  if (!ws || ws_bytes < pl.total || (reinterpret_cast<uintptr_t>(ws) & 255u)) return CONV2D_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const void *xsrc, *bhi, *blo;
  if ((rc = prep_forward_operands(g, x, w, ws, pl, &xsrc, &bhi, &blo, st))) return rc;
  float* scale = reinterpret_cast<float*>(region(ws, pl, R_FOLD));
  float* shift = scale + g.OC;
  LAUNCH("infer_fold", st,
         launch_infer_fold(bias, gamma, beta, running_mean, running_var, g.eps, g.norm, g.OC, scale, shift, st));
  if (g.norm == CONV2D_NORM_LAYER) {
    // `evaluate`, LAYER_NORM branch: the conv output is stored, then normalised with per-image
    // statistics computed on the fly (layer norm keeps no running statistics)
    void* ybuf = region(ws, pl, R_DC);
    float* rs = reinterpret_cast<float*>(region(ws, pl, R_PART));
    float* mean = shift + g.OC;
    float* istd = mean + g.N;
    RowStatLayout lay;
    if ((rc = run_fprop(g, dev, xsrc, bhi, blo, ybuf, nullptr, scale, shift, 0, nullptr, nullptr, rs, &lay, st)))
      return rc;
    LAUNCH("ln_stats_finalize", st,
           launch_ln_stats_finalize(rs, g.N, static_cast<long>(g.OH) * g.OW, lay.n_tiles, lay.halves, lay.BN,
                                    lay.hcols, g.OC, g.eps, mean, istd, st));
    LAUNCH("ln_apply", st, launch_bn_apply(g.dt, ybuf, y, pl.walk, mean, istd, gamma, beta, g.act, 1, st));
    return CONV2D_OK;
  }
  if (g.norm == CONV2D_NORM_GROUP) {
    // group norm at inference: the same per-(image, group) statistics of the stored conv output
    void* ybuf = region(ws, pl, R_DC);
    float* gp = reinterpret_cast<float*>(region(ws, pl, R_PART));
    float* mean = shift + g.OC;
    float* istd = mean + static_cast<size_t>(g.N) * g.groups;
    if ((rc = run_fprop(g, dev, xsrc, bhi, blo, ybuf, nullptr, scale, shift, 0, nullptr, nullptr, nullptr, nullptr,
                        st)))
      return rc;
    LAUNCH("gn_stats", st, launch_norm_stats(g.dt, ybuf, pl.walk, 1, gp, st));
    LAUNCH("gn_stats_finalize", st, launch_gn_stats_finalize(gp, pl.walk, g.eps, mean, istd, st));
    LAUNCH("gn_apply", st, launch_bn_apply(g.dt, ybuf, y, pl.walk, mean, istd, gamma, beta, g.act, 0, st));
    return CONV2D_OK;
  }
  return run_fprop(g, dev, xsrc, bhi, blo, y, nullptr, scale, shift, 1, nullptr, nullptr, nullptr, nullptr, st);
}

int conv2d_bwd(const conv2d_desc* desc, const void* x, const void* w, const float* gamma, const float* beta,
               const void* pre_act, const float* save_mean, const float* save_inv_std, const void* dy, void* dx,
               float* dw, float* dbias, float* dgamma, float* dbeta, void* ws, size_t ws_bytes, void* stream) {
  Geo g;
  int rc = make_geo(desc, &g);
  if (rc) return rc;
  REQ_PTR(pre_act); REQ_PTR(dy); OPT_PTR(dx); OPT_PTR(dw); OPT_PTR(dbias); OPT_PTR(dgamma); OPT_PTR(dbeta);
  if (!dx && !dw) return CONV2D_ERR_INVALID_ARG;
  if (dw && !dbias) return CONV2D_ERR_INVALID_ARG;
  if (dx) REQ_PTR(w);
  if (dw) REQ_PTR(x);
  const bool bn = g.norm == CONV2D_NORM_BATCH;
  const bool ln = g.norm == CONV2D_NORM_LAYER || g.norm == CONV2D_NORM_GROUP;  // per-(image, group) statistics
  if (bn || ln) {
    REQ_PTR(gamma); REQ_PTR(beta); REQ_PTR(save_mean); REQ_PTR(save_inv_std);
    if (static_cast<bool>(dgamma) != static_cast<bool>(dbeta)) return CONV2D_ERR_INVALID_ARG;
  }
  DevInfo* dev = nullptr;
  if ((rc = device_info(&dev))) return rc;
  Plan pl;
  plan_ws(g, CONV2D_OP_BWD, dev->sms, &pl);
  pl.walk.err = dev->err;
  pl.walk3.err = dev->err;
  if (!ws || ws_bytes < pl.total || (reinterpret_cast<uintptr_t>(ws) & 255u)) return CONV2D_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* dconv = region(ws, pl, R_DC);
  float* part = reinterpret_cast<float*>(region(ws, pl, R_PART));
  float* c12 = reinterpret_cast<float*>(region(ws, pl, R_C12));
  if (ln) {
    // per-channel sums of d_norm and d_norm * z (dbeta, dgamma) and, from the same image-aligned block
    // partials, the per-image sums of gamma * d_norm and gamma * d_norm * z
    LAUNCH("ln_bwd_reduce", st,
           launch_bn_bwd_reduce(g.dt, pre_act, dy, pl.walk, save_mean, save_inv_std, gamma, beta, g.act, part, 2,
                                st));
    LAUNCH("ln_bwd_finalize", st, launch_sum_finalize(part, pl.walk, 2, 0, c12, dbeta, dgamma, st));
    LAUNCH("ln_seg_finalize", st, launch_norm_seg_finalize(part, pl.walk, gamma, c12 + 2 * g.OC, st));
    LAUNCH("ln_bwd_dconv", st,
           launch_bn_bwd_apply(g.dt, pre_act, dy, pl.walk, g.OCp, save_mean, save_inv_std, gamma, beta, g.act, c12,
                               dconv, part, st));
  } else if (bn && pl.fused) {
    // d_conv is formed inside the dgrad and wgrad producers (bwd_fused): the reduce's third partial gives
    // dbias, and the finalize writes the per-channel terms of d_conv
    LAUNCH("bn_bwd_reduce", st,
           launch_bn_bwd_reduce(g.dt, pre_act, dy, pl.walk3, save_mean, save_inv_std, gamma, beta, g.act, part, 3,
                                st));
    LAUNCH("bn_bwd_finalize", st,
           launch_bn_bwd_fused_finalize(part, pl.walk3, save_mean, save_inv_std, gamma, beta, c12, dbeta, dgamma,
                                        dbias, c12 + 2 * g.OC, st));  // the terms of d_conv [4][OC] after c12
  } else if (bn) {
    // the reduce walks with three blocks per SM (its own block count; the partials are summed before the
    // d_conv pass reuses the buffer)
    LAUNCH("bn_bwd_reduce", st,
           launch_bn_bwd_reduce(g.dt, pre_act, dy, pl.walk3, save_mean, save_inv_std, gamma, beta, g.act, part, 2,
                                st));
    LAUNCH("bn_bwd_finalize", st, launch_sum_finalize(part, pl.walk3, 2, 0, c12, dbeta, dgamma, st));
    // evaluation mode (frozen statistics): d_conv = d_norm * gamma * inv_std, no projection terms
    LAUNCH("bn_bwd_dconv", st,
           launch_bn_bwd_apply(g.dt, pre_act, dy, pl.walk, g.OCp, save_mean, save_inv_std, gamma, beta, g.act,
                               g.bn_eval ? nullptr : c12, dconv, part, st));
  } else {
    LAUNCH("act_bwd_dconv", st, launch_act_bwd(g.dt, pre_act, dy, pl.walk, g.OCp, g.act, dconv, part, st));
  }
  // dbias = the sum of the d_conv pass's partials: in the split reduce's launch when dW is computed (the
  // partials stay untouched until then), else on its own (the fused backward has formed it already)
  const bool dbias_in_reduce = dbias && dw && !pl.fused;
  if (dbias && !dw && !pl.fused)
    LAUNCH("dbias_finalize", st, launch_sum_finalize(part, pl.walk, 1, 1, nullptr, dbias, nullptr, st));
  XfSrc xfs{pre_act, dy, c12 + 2 * g.OC};
  const XfSrc* xf = pl.fused ? &xfs : nullptr;
  if (pl.fused) dconv = nullptr;  // not formed
  if (dx && (rc = run_dgrad(g, dev, w, dconv, dx, ws, pl, st, xf))) return rc;
  if (dw) {
    const void* xsrc = x;
    if (g.pack_x) {
      void* xp = region(ws, pl, R_XP);
      LAUNCH("pack_x", st, launch_pack_channels(g.dt, x, xp, static_cast<long>(g.N) * g.H * g.W, g.IC, g.ICp, st));
      xsrc = xp;
    }
    if ((rc = run_wgrad(g, dev, xsrc, dconv, dw, ws, pl, st, xf, dbias_in_reduce ? part : nullptr, pl.walk.G,
                        dbias_in_reduce ? dbias : nullptr)))
      return rc;
  }
  return CONV2D_OK;
}

int conv2d_device_status(void* stream, int32_t* site) {
  DevInfo* dev = nullptr;
  int rc = device_info(&dev);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return CONV2D_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, dev->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return CONV2D_ERR_CUDA;
  if (site) *site = v;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(dev->err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return CONV2D_ERR_CUDA;
    return CONV2D_ERR_TIMEOUT;
  }
  return CONV2D_OK;
}

const char* conv2d_status_str(int status) {
  switch (status) {
    case CONV2D_OK: return "ok";
    case CONV2D_ERR_INVALID_ARG: return "invalid argument";
    case CONV2D_ERR_UNSUPPORTED: return "unsupported configuration";
    case CONV2D_ERR_WORKSPACE: return "workspace missing or too small";
    case CONV2D_ERR_CUDA: return "CUDA error";
    case CONV2D_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

int conv2d_prof_enable(int on) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = on != 0;
  return CONV2D_OK;
}

int conv2d_prof_read(const char** names, float* ms, int cap) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (cudaDeviceSynchronize() != cudaSuccess) return -1;
  int n = 0;
  for (int i = 0; i < g_prof_count && n < cap; ++i) {
    ProfRec& r = g_prof[(g_prof_head + i) % kProfCap];
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) t = -1.f;
    if (names) names[n] = r.name;
    if (ms) ms[n] = t;
    ++n;
  }
  g_prof_head = 0;
  g_prof_count = 0;
  return n;
}

}  // extern "C"
