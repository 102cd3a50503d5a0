// bn_kernels.cu - the bandwidth-bound steps of the conv2d training step:
// batch-, layer- and group-norm statistics, normalise + affine + activation,
// activation / norm backward (d_conv, dgamma, dbeta, dbias), weight
// preparation for the tensor-core GEMMs, and the split-K reduction of dW.
//
// Formulas: rl-tools "operations_generic.h" (`forward` BN training branch and
// Phase 3; `backward_full` training branch) and the per-channel kernels of
// "operations_cuda.h" (`bn_stats_training`, `bn_forward_affine`,
// `bn_training_backward`, `bias_backward_partial/finalize`). The layout work
// is different from those kernels: NHWC rows stream through shared memory
// (bulk copies) or are read with 16-byte vector loads, a thread keeps a fixed
// group of channels for its whole walk, and each block writes one partial per
// channel that a small finalize kernel merges in a fixed order
// (deterministic; fp32 with compensated sums or Chan merges, fp64 only where
// the work is a handful of operations). The batch variance is merged from
// per-tile (mean, M2) with Chan's formula, never E[x^2] - mean^2.
#include <algorithm>
#include <cmath>
#include <type_traits>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include "kernels.h"
#include "ptx.cuh"

namespace c2d {

namespace {

constexpr int kBlock = 256;
// Layers stored in bf16 take the fast activations (see act_f).
template <typename T>
constexpr bool kFastAct = std::is_same<T, __nv_bfloat16>::value;

template <int EC>
__device__ __forceinline__ void load_v(const float* p, float (&v)[EC]) {
  if constexpr (EC == 4) {
    const float4 t = __ldg(reinterpret_cast<const float4*>(p));
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
  } else {
#pragma unroll
    for (int e = 0; e < EC; ++e) v[e] = __ldg(p + e);
  }
}
template <int EC>
__device__ __forceinline__ void load_v(const __nv_bfloat16* p, float (&v)[EC]) {
  if constexpr (EC == 8) {
    const uint4 t = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
      const float2 f = __bfloat1622float2(h);
      v[2 * e] = f.x;
      v[2 * e + 1] = f.y;
    }
  } else {
#pragma unroll
    for (int e = 0; e < EC; ++e) v[e] = __bfloat162float(p[e]);
  }
}
template <int EC>
__device__ __forceinline__ void store_v(float* p, const float (&v)[EC]) {
  if constexpr (EC == 4) {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  } else {
#pragma unroll
    for (int e = 0; e < EC; ++e) p[e] = v[e];
  }
}
template <int EC>
__device__ __forceinline__ void store_v(__nv_bfloat16* p, const float (&v)[EC]) {
  if constexpr (EC == 8) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
      w[e] = *reinterpret_cast<uint32_t*>(&h);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
#pragma unroll
    for (int e = 0; e < EC; ++e) p[e] = __float2bfloat16_rn(v[e]);
  }
}

// Rows of a walk are grouped in segments of seg_rows rows (one segment for
// batch norm: every row; one per image for layer norm), each split over bps
// blocks of at most rpb rows, so that a block never straddles two segments.
// A reversed walk (rev != 0) maps launch block b to logical block G-1-b and
// visits its rows last to first: consecutive bandwidth-bound kernels walk in
// opposite directions, so each starts on the rows the previous one touched
// last, which are still in L2. Partials are indexed by the logical block.
struct SegRange {
  int seg, lb;
  long r0, r1;
};
__device__ __forceinline__ SegRange seg_range(long seg_rows, int bps, long rpb, int rev = 0) {
  SegRange r;
  r.lb = rev ? static_cast<int>(gridDim.x - 1 - blockIdx.x) : static_cast<int>(blockIdx.x);
  r.seg = r.lb / bps;
  const long sb = static_cast<long>(r.seg) * seg_rows;
  r.r0 = sb + static_cast<long>(r.lb % bps) * rpb;
  r.r1 = min(sb + seg_rows, r.r0 + rpb);
  return r;
}

// Index of the statistics of channel c in segment seg: per channel (cpg == 0, batch norm) or per
// group of cpg consecutive channels of one segment = image (layer norm: cpg = C; group norm: C/groups).
__device__ __forceinline__ int stat_index(int cpg, int seg, int c, int C) {
  return cpg ? seg * (C / cpg) + c / cpg : c;
}

// Thread geometry of a block walking [rows][C]: `tpr` threads share a row,
// each owning EC consecutive channels; `rpp` rows are in flight per pass.
struct Lane {
  int cg, tpr, rpp, rl, g0, seg;
  long r0, r1;
};
__device__ __forceinline__ Lane lane_of(long seg_rows, int bps, int Cw, int EC, long rpb) {
  Lane l;
  l.cg = Cw / EC;
  l.tpr = l.cg < kBlock ? l.cg : kBlock;
  l.rpp = kBlock / l.tpr;
  l.rl = threadIdx.x / l.tpr;
  l.g0 = threadIdx.x % l.tpr;
  const SegRange r = seg_range(seg_rows, bps, rpb);
  l.seg = r.seg;
  l.r0 = r.r0;
  l.r1 = r.r1;
  return l;
}

// ------------------------------------------------------------ BN statistics
// Pairwise Chan merge of (count, mean, M2): symmetric in its two operands, so both lanes of a
// shuffle pair reach the same result.
__device__ __forceinline__ void chan_merge(float& n, float& m, float& M, float nb, float mb, float Mb) {
  const float nn = n + nb;
  if (nn > 0.f) {
    const float d = mb - m;
    const float mm = (n * m + nb * mb) / nn;
    M = M + Mb + d * d * (n * nb / nn);
    m = mm;
    n = nn;
  }
}

// Merge of per-tile (count, mean, M2) partials [G][C][3] written by the fprop GEMM epilogue: one warp
// per channel; each lane combines every 32nd partial as sums shifted by its first partial's mean
// (exact for M2 up to rounding: sum(M2_b + n_b (mean_b - K)^2) - (sum n_b (mean_b - K))^2 / n), then
// a fixed-order shuffle tree of Chan merges. fp32 throughout (GB300's fp64 rate is low); the same
// order on every run.
__global__ void __launch_bounds__(128) bn_stats_finalize_kernel(const float* __restrict__ part, int G, int C,
                                                                float eps, float momentum, float* mean,
                                                                float* inv_std, float* rm, float* rv) {
  pdl_entry();
  const int c = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (c >= C) return;  // the whole warp
  float cnt = 0.f, K = 0.f, S1 = 0.f, S2 = 0.f;
#pragma unroll 4
  for (int b = lane; b < G; b += 32) {
    const float* q = part + (static_cast<size_t>(b) * C + c) * 3;
    const float nb = q[0], mb = q[1], Mb = q[2];
    if (nb == 0.f) continue;
    if (cnt == 0.f) K = mb;
    const float d = mb - K;
    S1 = fmaf(nb, d, S1);
    S2 += fmaf(nb * d, d, Mb);
    cnt += nb;
  }
  float m = cnt > 0.f ? K + S1 / cnt : 0.f;
  float M = cnt > 0.f ? fmaxf(S2 - S1 * (S1 / cnt), 0.f) : 0.f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float nb = __shfl_xor_sync(0xffffffffu, cnt, off);
    const float mb = __shfl_xor_sync(0xffffffffu, m, off);
    const float Mb = __shfl_xor_sync(0xffffffffu, M, off);
    chan_merge(cnt, m, M, nb, mb, Mb);
  }
  if (lane == 0) {
    const float var = cnt > 0.f ? M / cnt : 0.f;  // biased, as on the pages
    mean[c] = m;
    inv_std[c] = static_cast<float>(1.0 / sqrt(static_cast<double>(var) + static_cast<double>(eps)));
    rm[c] = (1.f - momentum) * rm[c] + momentum * m;
    rv[c] = (1.f - momentum) * rv[c] + momentum * var;
  }
}

// ------------------------------------------------------------ BN apply + act
// Statistics are per channel (batch norm, cpg == 0) or per image and channel group (layer / group norm).
template <typename T, int EC>
__global__ void __launch_bounds__(kBlock) bn_apply_kernel(const T* __restrict__ pre, T* __restrict__ y,
                                                          long seg_rows, int bps, int C, long rpb, int cpg,
                                                          const float* __restrict__ mean,
                                                          const float* __restrict__ inv_std,
                                                          const float* __restrict__ gamma,
                                                          const float* __restrict__ beta, int act) {
  pdl_entry();
  const Lane l = lane_of(seg_rows, bps, C, EC, rpb);
  if (l.rl >= l.rpp) return;
  for (int g = l.g0; g < l.cg; g += l.tpr) {
    float mu[EC], sc[EC], be[EC];
#pragma unroll
    for (int e = 0; e < EC; ++e) {
      const int c = g * EC + e;
      const int si = stat_index(cpg, l.seg, c, C);
      mu[e] = mean[si];
      sc[e] = gamma[c] * inv_std[si];
      be[e] = beta[c];
    }
    for (long r = l.r0 + l.rl; r < l.r1; r += l.rpp) {
      float v[EC];
      load_v<EC>(pre + r * C + g * EC, v);
#pragma unroll
      for (int e = 0; e < EC; ++e) v[e] = act_f(act, fmaf(v[e] - mu[e], sc[e], be[e]), kFastAct<T>);
      store_v<EC>(y + r * C + g * EC, v);
    }
  }
}

// ------------------------------------------------------------ per-channel statistics of a walk
// part[b][c][3] = (rows, mean, M2) of channel c over block b's rows (group-norm statistics of the
// stored pre-activations); per thread sums shifted by its first value of each channel.
template <typename T, int EC>
__global__ void __launch_bounds__(kBlock) norm_stats_kernel(const T* __restrict__ pre, long seg_rows, int bps,
                                                            int C, long rpb, float* __restrict__ part) {
  pdl_entry();
  __shared__ float s_n[kBlock], s_m[kBlock * EC], s_M[kBlock * EC];
  const Lane l = lane_of(seg_rows, bps, C, EC, rpb);
  for (int gb = 0; gb < l.cg; gb += l.tpr) {
    const int g = gb + l.g0;
    const bool active = g < l.cg && l.rl < l.rpp;
    float K[EC], s1[EC], s2[EC], nt = 0.f;
#pragma unroll
    for (int e = 0; e < EC; ++e) K[e] = s1[e] = s2[e] = 0.f;
    if (active) {
      for (long r = l.r0 + l.rl; r < l.r1; r += l.rpp) {
        float v[EC];
        load_v<EC>(pre + r * C + g * EC, v);
        if (nt == 0.f) {
#pragma unroll
          for (int e = 0; e < EC; ++e) K[e] = v[e];
        }
#pragma unroll
        for (int e = 0; e < EC; ++e) {
          const float d = v[e] - K[e];
          s1[e] += d;
          s2[e] = fmaf(d, d, s2[e]);
        }
        nt += 1.f;
      }
    }
    s_n[threadIdx.x] = nt;
#pragma unroll
    for (int e = 0; e < EC; ++e) {
      s_m[threadIdx.x * EC + e] = nt > 0.f ? K[e] + s1[e] / nt : 0.f;
      s_M[threadIdx.x * EC + e] = nt > 0.f ? fmaxf(s2[e] - s1[e] * (s1[e] / nt), 0.f) : 0.f;
    }
    __syncthreads();
    if (active && l.rl == 0) {
      for (int e = 0; e < EC; ++e) {
        float n = 0.f, m = 0.f, M = 0.f;
        for (int k = 0; k < l.rpp; ++k) {
          const int t = k * l.tpr + l.g0;
          const float nb = s_n[t];
          if (nb == 0.f) continue;
          const float nn = n + nb, d = s_m[t * EC + e] - m, f = nb / nn;
          m = fmaf(d, f, m);
          M += s_M[t * EC + e] + d * d * n * f;
          n = nn;
        }
        float* o = part + (static_cast<size_t>(blockIdx.x) * C + g * EC + e) * 3;
        o[0] = n;
        o[1] = m;
        o[2] = M;
      }
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------ BN backward
// part[b][c] = {sum d_norm, sum d_norm * z}, d_norm = act'(gamma z + beta) dy.
template <typename T, int EC>
__global__ void __launch_bounds__(kBlock) bn_bwd_reduce_kernel(const T* __restrict__ pre, const T* __restrict__ dy,
                                                               long seg_rows, int bps, int C, long rpb, int cpg,
                                                               const float* __restrict__ mean,
                                                               const float* __restrict__ inv_std,
                                                               const float* __restrict__ gamma,
                                                               const float* __restrict__ beta, int act,
                                                               float* __restrict__ part) {
  pdl_entry();
  __shared__ float s_a[kBlock * EC], s_b[kBlock * EC];
  const Lane l = lane_of(seg_rows, bps, C, EC, rpb);
  for (int gb = 0; gb < l.cg; gb += l.tpr) {
    const int g = gb + l.g0;
    const bool active = g < l.cg && l.rl < l.rpp;
    float a[EC], b[EC];
#pragma unroll
    for (int e = 0; e < EC; ++e) a[e] = b[e] = 0.f;
    if (active) {
      float mu[EC], is[EC], ga[EC], be[EC];
#pragma unroll
      for (int e = 0; e < EC; ++e) {
        const int c = g * EC + e;
        const int si = stat_index(cpg, l.seg, c, C);
        mu[e] = mean[si];
        is[e] = inv_std[si];
        ga[e] = gamma[c];
        be[e] = beta[c];
      }
      for (long r = l.r0 + l.rl; r < l.r1; r += l.rpp) {
        float v[EC], d[EC];
        load_v<EC>(pre + r * C + g * EC, v);
        load_v<EC>(dy + r * C + g * EC, d);
#pragma unroll
        for (int e = 0; e < EC; ++e) {
          const float z = (v[e] - mu[e]) * is[e];
          const float dn = dact_f(act, fmaf(ga[e], z, be[e]), kFastAct<T>) * d[e];
          a[e] += dn;
          b[e] = fmaf(dn, z, b[e]);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < EC; ++e) {
      s_a[threadIdx.x * EC + e] = a[e];
      s_b[threadIdx.x * EC + e] = b[e];
    }
    __syncthreads();
    if (active && l.rl == 0) {
      for (int e = 0; e < EC; ++e) {
        float sa = 0.f, sb = 0.f;
        for (int k = 0; k < l.rpp; ++k) {
          sa += s_a[(k * l.tpr + l.g0) * EC + e];
          sb += s_b[(k * l.tpr + l.g0) * EC + e];
        }
        float* o = part + (static_cast<size_t>(blockIdx.x) * C + g * EC + e) * 2;
        o[0] = sa;
        o[1] = sb;
      }
    }
    __syncthreads();
  }
}

// Normalisation coefficients of d_conv = inv_std * (gamma * d_norm - K1 - z * K2):
//   batch norm  K1 = gamma * c1[c] / n,   K2 = gamma * c2[c] / n    (n = rows; c12 = [C][2] sums)
//   layer / group norm  K1 = s1[si] / M,  K2 = s2[si] / M  (si = stat_index, M = seg_rows * cpg; sums
//               of gamma * d_norm and gamma * d_norm * z per image and group, after the channel sums: c12 + 2C)
//   no c12      evaluation-mode batch norm, no projection terms.
__device__ __forceinline__ void norm_bwd_coef(const float* c12, int cpg, int seg, int c, int C, float ga,
                                              long seg_rows, float& k1, float& k2) {
  if (!c12) {
    k1 = k2 = 0.f;
  } else if (cpg) {
    const int si = stat_index(cpg, seg, c, C);
    const float inv_m = 1.f / static_cast<float>(seg_rows * cpg);
    k1 = c12[2 * C + 2 * si] * inv_m;
    k2 = c12[2 * C + 2 * si + 1] * inv_m;
  } else {
    const float inv_n = 1.f / static_cast<float>(seg_rows);
    k1 = ga * c12[2 * c] * inv_n;
    k2 = ga * c12[2 * c + 1] * inv_n;
  }
}

// part[b][c] = sum d_conv. MODE 0: batch / layer norm; MODE 1: no norm (d_conv = act'(pre) * dy).
template <typename T, int EC, int MODE>
__global__ void __launch_bounds__(kBlock) dconv_kernel(const T* __restrict__ pre, const T* __restrict__ dy,
                                                       long seg_rows, int bps, int C, int Cp, long rpb, int cpg,
                                                       const float* __restrict__ mean,
                                                       const float* __restrict__ inv_std,
                                                       const float* __restrict__ gamma,
                                                       const float* __restrict__ beta, int act,
                                                       const float* __restrict__ c12, T* __restrict__ dconv,
                                                       float* __restrict__ part) {
  pdl_entry();
  __shared__ float s_a[kBlock * EC];
  // the walk covers Cp channels so that padded channels of d_conv get zeros
  const Lane l = lane_of(seg_rows, bps, Cp, EC, rpb);
  for (int gb = 0; gb < l.cg; gb += l.tpr) {
    const int g = gb + l.g0;
    const bool active = g < l.cg && l.rl < l.rpp;
    const bool real = g * EC < C;  // EC divides C whenever EC > 1
    float a[EC];
#pragma unroll
    for (int e = 0; e < EC; ++e) a[e] = 0.f;
    if (active) {
      float mu[EC], is[EC], ga[EC], be[EC], k1[EC], k2[EC];
#pragma unroll
      for (int e = 0; e < EC; ++e) {
        const int c = real ? g * EC + e : 0;
        if (MODE == 0) {
          const int si = stat_index(cpg, l.seg, c, C);
          mu[e] = mean[si];
          is[e] = inv_std[si];
          ga[e] = gamma[c];
          be[e] = beta[c];
          norm_bwd_coef(c12, cpg, l.seg, c, C, ga[e], seg_rows, k1[e], k2[e]);
        }
      }
      for (long r = l.r0 + l.rl; r < l.r1; r += l.rpp) {
        float o[EC];
        if (real) {
          float v[EC], d[EC];
          load_v<EC>(pre + r * C + g * EC, v);
          load_v<EC>(dy + r * C + g * EC, d);
#pragma unroll
          for (int e = 0; e < EC; ++e) {
            if (MODE == 0) {
              const float z = (v[e] - mu[e]) * is[e];
              const float dn = dact_f(act, fmaf(ga[e], z, be[e]), kFastAct<T>) * d[e];
              o[e] = is[e] * (ga[e] * dn - k1[e] - z * k2[e]);
            } else {
              o[e] = dact_f(act, v[e], kFastAct<T>) * d[e];
            }
            a[e] += o[e];
          }
        } else {
#pragma unroll
          for (int e = 0; e < EC; ++e) o[e] = 0.f;
        }
        store_v<EC>(dconv + r * Cp + g * EC, o);
      }
    }
#pragma unroll
    for (int e = 0; e < EC; ++e) s_a[threadIdx.x * EC + e] = a[e];
    __syncthreads();
    if (active && real && l.rl == 0) {
      for (int e = 0; e < EC; ++e) {
        float sa = 0.f;
        for (int k = 0; k < l.rpp; ++k) sa += s_a[(k * l.tpr + l.g0) * EC + e];
        part[static_cast<size_t>(blockIdx.x) * C + g * EC + e] = sa;
      }
    }
    __syncthreads();
  }
}

__device__ __forceinline__ void kahan_add(float& s, float& comp, float x) {
  const float y = x - comp;
  const float t = s + y;
  comp = (t - s) - y;
  s = t;
}

// Per-channel sums of per-block partials [G][C][nv] (nv <= 3) by one block of 128 or 256 threads:
// compensated fp32 sums per thread over every blockDim-th partial, fp64 shuffle trees within the warps and
// the warp totals added in a fixed order (the same result on every run). Block-collective; the totals are
// valid in thread 0.
__device__ __forceinline__ void channel_sums(const float* __restrict__ part, int G, int C, int nv, int c,
                                             double (&tot)[3]) {
  __shared__ double s_w[3][8];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  float a[3] = {0.f, 0.f, 0.f}, ca[3] = {0.f, 0.f, 0.f};
#pragma unroll 4
  for (int k = threadIdx.x; k < G; k += blockDim.x) {
    const float* p = part + (static_cast<size_t>(k) * C + c) * nv;
    kahan_add(a[0], ca[0], p[0]);
    if (nv > 1) kahan_add(a[1], ca[1], p[1]);
    if (nv > 2) kahan_add(a[2], ca[2], p[2]);
  }
#pragma unroll
  for (int v = 0; v < 3; ++v) {
    double d = static_cast<double>(a[v]) - static_cast<double>(ca[v]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) d += __shfl_xor_sync(0xffffffffu, d, off);
    if (lane == 0) s_w[v][w] = d;
  }
  __syncthreads();
#pragma unroll
  for (int v = 0; v < 3; ++v) {
    tot[v] = (s_w[v][0] + s_w[v][1]) + (s_w[v][2] + s_w[v][3]);
    if (nw == 8) tot[v] += (s_w[v][4] + s_w[v][5]) + (s_w[v][6] + s_w[v][7]);
  }
}

// Blocks past the split reduce's own (blockIdx.x >= nb) sum the dbias partials bpart[bG][C] of channel
// blockIdx.x - nb into dbias (the dbias finalize, folded into the last launch of the backward). Returns
// true for those blocks.
__device__ __forceinline__ bool dbias_block(int nb, const float* __restrict__ bpart, int bG, int C, float* dbias) {
  if (static_cast<int>(blockIdx.x) < nb) return false;
  const int c = blockIdx.x - nb;
  double t[3];
  channel_sums(bpart, bG, C, 1, c, t);
  if (threadIdx.x == 0) dbias[c] += static_cast<float>(t[0]);
  return true;
}

// mode 0: c12 = (sum d_norm, sum d_norm z), dbeta += first, dgamma += second; mode 1: dbias += the sum.
__global__ void __launch_bounds__(128) sum_finalize_kernel(const float* __restrict__ part, int G, int C, int nv,
                                                           int mode, float* c12, float* acc0, float* acc1) {
  pdl_entry();
  const int c = blockIdx.x;
  double t[3];
  channel_sums(part, G, C, nv, c, t);
  if (threadIdx.x == 0) {
    if (mode == 0) {
      c12[2 * c] = static_cast<float>(t[0]);
      c12[2 * c + 1] = static_cast<float>(t[1]);
      if (acc0) acc0[c] += static_cast<float>(t[0]);  // dbeta
      if (acc1) acc1[c] += static_cast<float>(t[1]);  // dgamma
    } else {
      if (acc0) acc0[c] += static_cast<float>(t[0]);  // dbias
    }
  }
}

// Batch norm (training statistics) with d_conv formed inside the GEMM producers: from the backward
// reduce's partials (sum d_norm, sum d_norm z, sum (x - mean)) per channel, c12 and dbeta / dgamma as in
// sum_finalize_kernel mode 0, and:
//   the terms of d_conv tbl[4][C] = (G, B', Q, S'): with G = gamma inv_std and k1, k2 as norm_bwd_coef
//   forms them, t = gamma z + beta = G x + B' (B' = beta - G mean) and d_conv = inv_std (gamma d_norm - k1
//   - z k2) = G d_norm + Q x + S' (Q = -inv_std^2 k2, S' = -inv_std k1 - Q mean); B' and S' in fp64;
//   dbias = sum over pixels of d_conv without the d_conv tensor: inv_std (gamma sum d_norm - n k1) - inv_std
//   k2 sum z, whose first term vanishes by the definition of k1, so dbias += -inv_std^2 k2 sum (x - mean).
__global__ void __launch_bounds__(128) bn_bwd_fused_finalize_kernel(const float* __restrict__ part, int G, int C,
                                                                    long n, const float* __restrict__ mean,
                                                                    const float* __restrict__ inv_std,
                                                                    const float* __restrict__ gamma,
                                                                    const float* __restrict__ beta, float* c12,
                                                                    float* dbeta, float* dgamma, float* dbias,
                                                                    float* tbl) {
  pdl_entry();
  const int c = blockIdx.x;
  double t[3];
  channel_sums(part, G, C, 3, c, t);
  if (threadIdx.x == 0) {
    const float s1 = static_cast<float>(t[0]), s2 = static_cast<float>(t[1]);
    c12[2 * c] = s1;
    c12[2 * c + 1] = s2;
    if (dbeta) dbeta[c] += s1;
    if (dgamma) dgamma[c] += s2;
    const float ga = gamma[c], is = inv_std[c];
    float k1, k2;
    norm_bwd_coef(c12, 0, 0, c, C, ga, n, k1, k2);
    const double g = static_cast<double>(ga) * is, q = -static_cast<double>(is) * is * k2;
    tbl[c] = static_cast<float>(g);
    tbl[C + c] = static_cast<float>(beta[c] - g * mean[c]);
    tbl[2 * C + c] = static_cast<float>(q);
    tbl[3 * C + c] = static_cast<float>(-static_cast<double>(is) * k1 - q * mean[c]);
    if (dbias) dbias[c] += static_cast<float>(q * t[2]);
  }
}

// ------------------------------------------------------------ layout prep
template <typename T>
__global__ void pack_channels_kernel(const T* __restrict__ src, T* __restrict__ dst, long rows, int C, int Cp) {
  pdl_entry();
  const long total = rows * Cp;
  for (long i = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    const long r = i / Cp;
    const int c = static_cast<int>(i - r * Cp);
    dst[i] = c < C ? src[r * C + c] : T(0.f);
  }
}

// B[oc][tap][icp] from W[oc][tap][ic]; fp32: tf32 hi / lo split.
template <typename T>
__global__ void prep_fprop_weights_kernel(const T* __restrict__ w, T* __restrict__ bhi, float* __restrict__ blo,
                                          int OC, int taps, int IC, int ICp) {
  pdl_entry();
  const long total = static_cast<long>(OC) * taps * ICp;
  for (long i = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    const int ic = static_cast<int>(i % ICp);
    const long ot = i / ICp;
    const T v = ic < IC ? w[ot * IC + ic] : T(0.f);
    if constexpr (sizeof(T) == 4) {
      uint32_t hi, lo;
      split_tf32(static_cast<float>(v), hi, lo);
      reinterpret_cast<uint32_t*>(bhi)[i] = hi;
      reinterpret_cast<uint32_t*>(blo)[i] = lo;
    } else {
      bhi[i] = v;
    }
  }
}

// Column-form dgrad weights: B[(tap, icp)][oc], K = OCp, the transpose of W[oc][tap][ic] (zero in the
// padded ic and oc positions); 3xTF32 splits into hi / lo.
template <typename T>
__global__ void prep_col2im_weights_kernel(const T* __restrict__ w, T* __restrict__ bhi, float* __restrict__ blo,
                                           int OC, int taps, int IC, int ICp, int OCp) {
  pdl_entry();
  const long total = static_cast<long>(taps) * ICp * OCp;
  for (long i = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    const int oc = static_cast<int>(i % OCp);
    const long r = i / OCp;
    const int ic = static_cast<int>(r % ICp), tap = static_cast<int>(r / ICp);
    const T v = (oc < OC && ic < IC) ? w[(static_cast<long>(oc) * taps + tap) * IC + ic] : T(0.f);
    if constexpr (sizeof(T) == 4) {
      uint32_t hi, lo;
      split_tf32(static_cast<float>(v), hi, lo);
      reinterpret_cast<uint32_t*>(bhi)[i] = hi;
      reinterpret_cast<uint32_t*>(blo)[i] = lo;
    } else {
      bhi[i] = v;
    }
  }
}

// dX from the column form dcol[(n, oh, ow)][(kh, kw, icp)] = sum_oc d_conv * W: each input pixel sums
// the kernel taps whose window covers it (`backward_full`'s scatter of d_conv * W, gathered per dX
// element), in a fixed (kh, kw) order.
template <typename T, int EC>
__global__ void col2im_kernel(const T* __restrict__ dcol, T* __restrict__ dx, int N, int H, int W, int IC, int ICp,
                              int OH, int OW, int KH, int KW, int S, int P) {
  pdl_entry();
  const int groups = IC / EC;
  const long total = static_cast<long>(N) * H * W * groups;
  const int taps_icp = KH * KW * ICp;
  for (long i = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    const int g = static_cast<int>(i % groups);
    const long pix = i / groups;
    const int iw = static_cast<int>(pix % W);
    const long t = pix / W;
    const int ih = static_cast<int>(t % H);
    const int n = static_cast<int>(t / H);
    float acc[EC];
#pragma unroll
    for (int e = 0; e < EC; ++e) acc[e] = 0.f;
    for (int kh = (ih + P) % S; kh < KH; kh += S) {
      const int oh = (ih + P - kh) / S;
      if (oh < 0) break;
      if (oh >= OH) continue;
      for (int kw = (iw + P) % S; kw < KW; kw += S) {
        const int ow = (iw + P - kw) / S;
        if (ow < 0) break;
        if (ow >= OW) continue;
        float v[EC];
        load_v<EC>(dcol + (static_cast<size_t>(n * OH + oh) * OW + ow) * taps_icp + (kh * KW + kw) * ICp + g * EC,
                   v);
#pragma unroll
        for (int e = 0; e < EC; ++e) acc[e] += v[e];
      }
    }
    store_v<EC>(dx + pix * IC + g * EC, acc);
  }
}

// dgrad weight matrix B[icp][col]; for phase ph the columns (t,u,oc) hold
// W[oc][rh + S*t][rw + S*u][ic].
template <typename T>
__global__ void prep_dgrad_weights_kernel(const T* __restrict__ w, T* __restrict__ bhi, float* __restrict__ blo,
                                          int OC, int KH, int KW, int IC, int ICp, int OCp, int S, int Kd,
                                          const DgradWeightTable t) {
  pdl_entry();
  const long total = static_cast<long>(ICp) * Kd;
  for (long i = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    const int ic = static_cast<int>(i / Kd);
    const int col = static_cast<int>(i - static_cast<long>(ic) * Kd);
    int ph = 0;
    while (ph + 1 < t.n && t.col_off[ph + 1] <= col) ++ph;
    const int local = col - t.col_off[ph];
    const int oc = local % OCp;
    const int tap = local / OCp;
    int tt = tap / t.Tw[ph], uu = tap % t.Tw[ph];
    if (t.flip) {
      tt = t.Th[ph] - 1 - tt;
      uu = t.Tw[ph] - 1 - uu;
    }
    const int kh = t.rh[ph] + S * tt, kw = t.rw[ph] + S * uu;
    T v = T(0.f);
    if (ic < IC && oc < OC && tt < t.Th[ph] && kh < KH && kw < KW)
      v = w[((static_cast<long>(oc) * KH + kh) * KW + kw) * IC + ic];
    if constexpr (sizeof(T) == 4) {
      uint32_t hi, lo;
      split_tf32(static_cast<float>(v), hi, lo);
      reinterpret_cast<uint32_t*>(bhi)[i] = hi;
      reinterpret_cast<uint32_t*>(blo)[i] = lo;
    } else {
      bhi[i] = v;
    }
  }
}

// Phase-merged dgrad weights (every stride phase has Th x Tw taps, KH = S Th, KW = S Tw, pad a multiple of
// S): row (ph_h * S + ph_w) * ICp + ic, column (t * Tw + u) * OCp + oc holds W[oc][ph_h + S (Th-1-t)]
// [ph_w + S (Tw-1-u)][ic] (taps reversed: the im2col window of d_conv starts Th-1, Tw-1 pixels up-left).
template <typename T>
__global__ void prep_dgrad_merged_weights_kernel(const T* __restrict__ w, T* __restrict__ bhi,
                                                 float* __restrict__ blo, int OC, int KH, int KW, int IC, int ICp,
                                                 int OCp, int S) {
  pdl_entry();
  const int Th = KH / S, Tw = KW / S;
  const long Kd = static_cast<long>(Th) * Tw * OCp;
  const long total = static_cast<long>(S) * S * ICp * Kd;
  for (long i = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    const long row = i / Kd;
    const int col = static_cast<int>(i - row * Kd);
    const int ic = static_cast<int>(row % ICp);
    const int ph = static_cast<int>(row / ICp);
    const int ph_h = ph / S, ph_w = ph % S;
    const int oc = col % OCp, tap = col / OCp;
    const int kh = ph_h + S * (Th - 1 - tap / Tw), kw = ph_w + S * (Tw - 1 - tap % Tw);
    T v = T(0.f);
    if (ic < IC && oc < OC) v = w[((static_cast<long>(oc) * KH + kh) * KW + kw) * IC + ic];
    if constexpr (sizeof(T) == 4) {
      uint32_t hi, lo;
      split_tf32(static_cast<float>(v), hi, lo);
      reinterpret_cast<uint32_t*>(bhi)[i] = hi;
      reinterpret_cast<uint32_t*>(blo)[i] = lo;
    } else {
      bhi[i] = v;
    }
  }
}

// dW[oc][tap][ic] += sum over splits of partial[s][oc][tap*ICp + ic] (fixed order: deterministic), one
// thread per item over all splits: the form for a few splits (see launch_wgrad_reduce).
__global__ void wgrad_reduce_serial_kernel(const float* __restrict__ partial, int splits, int OC, int taps, int ICp,
                                           int IC, float* __restrict__ dw, int nb, const float* __restrict__ bpart,
                                           int bG, float* dbias) {
  pdl_entry();
  if (dbias_block(nb, bpart, bG, OC, dbias)) return;
  // V consecutive input channels per thread (4 when IC == ICp is a multiple of 4: 16-byte loads and
  // stores), each summed over the splits with compensated (Kahan) fp32 summation in split order
  // (fp64 is slow on this part); the loads of eight splits are issued before their sums
  const int V = (IC == ICp && IC % 4 == 0) ? 4 : 1;
  const long total = static_cast<long>(OC) * taps * IC / V;
  const long Mk = static_cast<long>(taps) * ICp;
  const long stride = static_cast<long>(OC) * Mk;
  for (long i = blockIdx.x * static_cast<long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long>(nb) * blockDim.x) {
    const long e = i * V;  // first dw element of this thread
    const int ic = static_cast<int>(e % IC);
    const long ot = e / IC;
    const int tap = static_cast<int>(ot % taps);
    const int oc = static_cast<int>(ot / taps);
    const float* q = partial + static_cast<long>(oc) * Mk + static_cast<long>(tap) * ICp + ic;
    if (V == 4) {
      float4 s = make_float4(0.f, 0.f, 0.f, 0.f), c = s;
      auto add = [](float& sum, float& comp, float x) {
        const float y = x - comp;
        const float t = sum + y;
        comp = (t - sum) - y;
        sum = t;
      };
      int k = 0;
      for (; k + 8 <= splits; k += 8) {
        float4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = *reinterpret_cast<const float4*>(q + (k + j) * stride);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          add(s.x, c.x, v[j].x);
          add(s.y, c.y, v[j].y);
          add(s.z, c.z, v[j].z);
          add(s.w, c.w, v[j].w);
        }
      }
      for (; k < splits; ++k) {
        const float4 v = *reinterpret_cast<const float4*>(q + k * stride);
        add(s.x, c.x, v.x);
        add(s.y, c.y, v.y);
        add(s.z, c.z, v.z);
        add(s.w, c.w, v.w);
      }
      float4* d = reinterpret_cast<float4*>(dw + e);
      float4 o = *d;
      o.x += s.x;
      o.y += s.y;
      o.z += s.z;
      o.w += s.w;
      *d = o;
    } else {
      float s = 0.f, comp = 0.f;
      int k = 0;
      for (; k + 8 <= splits; k += 8) {
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = q[(k + j) * stride];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float yk = v[j] - comp;
          const float t = s + yk;
          comp = (t - s) - yk;
          s = t;
        }
      }
      for (; k < splits; ++k) {
        const float yk = q[k * stride] - comp;
        const float t = s + yk;
        comp = (t - s) - yk;
        s = t;
      }
      dw[e] += s;
    }
  }
}

// dW[oc][tap][ic] += sum over splits of partial[s][oc][tap*ICp + ic] (fixed order: deterministic).
// A block holds 32 items (V consecutive input channels each: 4 when IC == ICp is a multiple of 4, for
// 16-byte loads and stores) and kRedGroups warps: warp g sums splits g, g + kRedGroups, ... of its
// lane's item with compensated (Kahan) fp32 sums in split order (fp64 is slow on this part), so that a
// thread's chain of dependent loads is splits / kRedGroups long; warp 0 then adds the group sums in
// group order. 32-bit index arithmetic: the layer limits keep OC * taps * ICp below 2^30.
constexpr int kRedGroups = 8;
constexpr int kRedSerialMax = 48;  // split counts below this take wgrad_reduce_serial_kernel
template <int V>
__global__ void __launch_bounds__(32 * kRedGroups) wgrad_reduce_kernel(const float* __restrict__ partial, int splits,
                                                                      int OC, int taps, int ICp, int IC,
                                                                      float* __restrict__ dw, int nb,
                                                                      const float* __restrict__ bpart, int bG,
                                                                      float* dbias) {
  pdl_entry();
  if (dbias_block(nb, bpart, bG, OC, dbias)) return;
  using VT = typename std::conditional<V == 4, float4, float>::type;
  __shared__ VT s_sum[kRedGroups][32];
  const int lane = threadIdx.x & 31, grp = threadIdx.x >> 5;
  const int total = OC * taps * IC / V;
  const int item = blockIdx.x * 32 + lane;
  const long stride = static_cast<long>(OC) * taps * ICp;
  float sum[V], comp[V];
#pragma unroll
  for (int j = 0; j < V; ++j) sum[j] = comp[j] = 0.f;
  int e = 0;
  if (item < total) {
    e = item * V;  // first dw element of this item
    const int ot = e / IC;
    const int ic = e - ot * IC;
    const int oc = ot / taps;
    const int tap = ot - oc * taps;
    const float* q = partial + oc * taps * ICp + tap * ICp + ic;
    int k = grp;
    // four loads in flight per thread before their sums
    for (; k + 3 * kRedGroups < splits; k += 4 * kRedGroups) {
      VT v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = *reinterpret_cast<const VT*>(q + (k + u * kRedGroups) * stride);
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int j = 0; j < V; ++j) kahan_add(sum[j], comp[j], reinterpret_cast<const float*>(&v[u])[j]);
    }
    for (; k < splits; k += kRedGroups) {
      const VT v = *reinterpret_cast<const VT*>(q + k * stride);
#pragma unroll
      for (int j = 0; j < V; ++j) kahan_add(sum[j], comp[j], reinterpret_cast<const float*>(&v)[j]);
    }
  }
  {
    VT t;
#pragma unroll
    for (int j = 0; j < V; ++j) reinterpret_cast<float*>(&t)[j] = sum[j] - comp[j];
    s_sum[grp][lane] = t;
  }
  __syncthreads();
  if (grp == 0 && item < total) {
    float acc[V], cacc[V];
#pragma unroll
    for (int j = 0; j < V; ++j) acc[j] = cacc[j] = 0.f;
    for (int g = 0; g < kRedGroups; ++g) {
      const VT t = s_sum[g][lane];
#pragma unroll
      for (int j = 0; j < V; ++j) kahan_add(acc[j], cacc[j], reinterpret_cast<const float*>(&t)[j]);
    }
    VT* d = reinterpret_cast<VT*>(dw + e);
    VT o = *d;
#pragma unroll
    for (int j = 0; j < V; ++j) reinterpret_cast<float*>(&o)[j] += acc[j];
    *d = o;
  }
}

// Batch norm in evaluation mode inside training: the saved statistics are the
// running ones (`forward` with mode::Evaluation), nothing is updated.
__global__ void bn_eval_stats_kernel(const float* rm, const float* rv, float eps, int C, float* mean,
                                     float* inv_std) {
  pdl_entry();
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= C) return;
  mean[c] = rm[c];
  inv_std[c] = static_cast<float>(1.0 / sqrt(static_cast<double>(rv[c]) + eps));
}

// Inference epilogue constants: v = acc*scale + shift folds bias and the
// running-statistics normalisation (`evaluate`, BN branch).
__global__ void infer_fold_kernel(const float* bias, const float* gamma, const float* beta, const float* rm,
                                  const float* rv, float eps, int norm, int OC, float* scale, float* shift) {
  pdl_entry();
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= OC) return;
  const float b = bias ? bias[c] : 0.f;
  if (norm == 1) {
    const float is = static_cast<float>(1.0 / sqrt(static_cast<double>(rv[c]) + eps));
    const float sc = gamma[c] * is;
    scale[c] = sc;
    shift[c] = fmaf(b - rm[c], sc, beta[c]);
  } else {
    scale[c] = 1.f;
    shift[c] = b;
  }
}

// ------------------------------------------------------------ layer norm
// Per-image statistics (`forward` LAYER_NORM branch, over OH*OW*OC of the
// stored pre-activations) from the per-pixel (mean, M2) partials of the
// fprop epilogue, one per column tile and column half (halves = 1 or 2; half
// 0 holds the first hcols columns of the tile): block n merges the partials
// of image n, in fp32 per thread (Chan) and then in fp64 in a fixed tree.
__global__ void __launch_bounds__(256) ln_stats_finalize_kernel(const float* __restrict__ rs, int n_tiles,
                                                                int halves, int BN, int hcols, int OC, long hw,
                                                                float eps, float* mean, float* inv_std) {
  pdl_entry();
  __shared__ float s_n[8], s_m[8], s_M[8];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int per_pix = n_tiles * halves;
  const long n_ent = hw * per_pix;
  const float* base = rs + static_cast<size_t>(blockIdx.x) * n_ent * 2;
  // per thread: sums shifted by the thread's first partial mean K (no division per partial),
  // S1 = sum n_j (m_j - K), S2 = sum M2_j + n_j (m_j - K)^2
  float cnt = 0.f, K = 0.f, S1 = 0.f, S2 = 0.f;
  for (long e = threadIdx.x; e < n_ent; e += 256) {
    const int j = static_cast<int>(e % per_pix);
    const int t = j / halves, h = j % halves;
    const int c0 = t * BN + h * hcols;
    const int c1 = min(OC, t * BN + ((h + 1 == halves) ? BN : hcols));
    if (c1 <= c0) continue;  // a half with no channel of the layer
    const float nb = static_cast<float>(c1 - c0);
    const float mb = base[2 * e], Mb = base[2 * e + 1];
    if (cnt == 0.f) K = mb;
    const float d = mb - K;
    S1 = fmaf(nb, d, S1);
    S2 += fmaf(nb * d, d, Mb);
    cnt += nb;
  }
  float m = cnt > 0.f ? K + S1 / cnt : 0.f;
  float M = cnt > 0.f ? fmaxf(S2 - S1 * (S1 / cnt), 0.f) : 0.f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float nb = __shfl_xor_sync(0xffffffffu, cnt, off);
    const float mb = __shfl_xor_sync(0xffffffffu, m, off);
    const float Mb = __shfl_xor_sync(0xffffffffu, M, off);
    const float nn = cnt + nb;
    if (nn > 0.f) {  // symmetric in the two operands: both lanes of a pair agree
      const float d = mb - m;
      const float mm = (cnt * m + nb * mb) / nn;
      M = M + Mb + d * d * (cnt * nb / nn);
      m = mm;
      cnt = nn;
    }
  }
  if (lane == 0) {
    s_n[w] = cnt;
    s_m[w] = m;
    s_M[w] = M;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double n = 0.0, mu = 0.0, M2 = 0.0;
    for (int k = 0; k < 8; ++k) {
      const double nb = s_n[k];
      if (nb == 0.0) continue;
      const double nn = n + nb, d = s_m[k] - mu;
      mu += d * nb / nn;
      M2 += s_M[k] + d * d * n * nb / nn;
      n = nn;
    }
    const double var = n > 0 ? M2 / n : 0.0;  // biased
    mean[blockIdx.x] = static_cast<float>(mu);
    inv_std[blockIdx.x] = static_cast<float>(1.0 / sqrt(var + static_cast<double>(eps)));
  }
}

// Warps per output of the per-(image, group) finalize kernels: more warps when an output merges many
// partials (layer norm: every channel of an image), one when it merges few (group norm).
static int finalize_wpo(long n_ent) { return n_ent >= 1024 ? 4 : (n_ent >= 256 ? 2 : 1); }

// Per-(image, group) sums of gamma * d_norm and gamma * d_norm * z (`backward_full` training branch
// with NORM_DIM = batch for layer norm; Phase 2 of the GroupNorm backward shader for group norm) from
// the per-block, per-channel partials part[b][c][2] of an image-aligned walk (bps blocks per image).
// wpo warps per output s = n * groups + g: fp32 sums per lane, a fixed shuffle tree per warp, the wpo
// warp sums added in a fixed order; written to out[2s], out[2s+1].
__global__ void __launch_bounds__(128) norm_seg_finalize_kernel(const float* __restrict__ part, int bps, int C,
                                                                int cpg, int n_out, int wpo,
                                                                const float* __restrict__ gamma, float* out) {
  pdl_entry();
  __shared__ float s_a[4], s_b[4];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.x * (4 / wpo) + w / wpo, sub = w % wpo;
  const int groups = C / cpg;
  const int n = s / groups, g = s % groups;
  const long n_ent = static_cast<long>(bps) * cpg;
  float a = 0.f, b = 0.f;
  if (s < n_out) {
    for (long k = sub * 32 + lane; k < n_ent; k += 32 * wpo) {
      const int j = static_cast<int>(k / cpg), c = g * cpg + static_cast<int>(k % cpg);
      const float* q = part + (static_cast<size_t>(n * bps + j) * C + c) * 2;
      a = fmaf(gamma[c], q[0], a);
      b = fmaf(gamma[c], q[1], b);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, off);
    b += __shfl_xor_sync(0xffffffffu, b, off);
  }
  if (lane == 0) {
    s_a[w] = a;
    s_b[w] = b;
  }
  __syncthreads();
  if (s < n_out && sub == 0 && lane == 0) {
    float ta = 0.f, tb = 0.f;
    for (int k = 0; k < wpo; ++k) {
      ta += s_a[w + k];
      tb += s_b[w + k];
    }
    out[2 * s] = ta;
    out[2 * s + 1] = tb;
  }
}

// Group-norm statistics per (image, group) from the per-block, per-channel (count, mean, M2) partials
// part[b][c][3] of an image-aligned walk over the stored pre-activations. wpo warps per output
// s = n * groups + g: per lane sums shifted by its first partial mean (no division per partial), a
// fixed Chan tree over the lanes, then over the wpo warps.

__global__ void __launch_bounds__(128) gn_stats_finalize_kernel(const float* __restrict__ part, int bps, int C,
                                                                int cpg, int n_out, int wpo, float eps, float* mean,
                                                                float* inv_std) {
  pdl_entry();
  __shared__ float s_n[4], s_m[4], s_M[4];
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.x * (4 / wpo) + w / wpo, sub = w % wpo;
  const int groups = C / cpg;
  const int n = s / groups, g = s % groups;
  const long n_ent = static_cast<long>(bps) * cpg;
  float cnt = 0.f, K = 0.f, S1 = 0.f, S2 = 0.f;
  if (s < n_out) {
    for (long k = sub * 32 + lane; k < n_ent; k += 32 * wpo) {
      const int j = static_cast<int>(k / cpg), c = g * cpg + static_cast<int>(k % cpg);
      const float* q = part + (static_cast<size_t>(n * bps + j) * C + c) * 3;
      const float nb = q[0];
      if (nb == 0.f) continue;
      if (cnt == 0.f) K = q[1];
      const float d = q[1] - K;
      S1 = fmaf(nb, d, S1);
      S2 += fmaf(nb * d, d, q[2]);
      cnt += nb;
    }
  }
  float m = cnt > 0.f ? K + S1 / cnt : 0.f;
  float M = cnt > 0.f ? fmaxf(S2 - S1 * (S1 / cnt), 0.f) : 0.f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float nb = __shfl_xor_sync(0xffffffffu, cnt, off);
    const float mb = __shfl_xor_sync(0xffffffffu, m, off);
    const float Mb = __shfl_xor_sync(0xffffffffu, M, off);
    chan_merge(cnt, m, M, nb, mb, Mb);
  }
  if (lane == 0) {
    s_n[w] = cnt;
    s_m[w] = m;
    s_M[w] = M;
  }
  __syncthreads();
  if (s < n_out && sub == 0 && lane == 0) {
    float tn = 0.f, tm = 0.f, tM = 0.f;
    for (int k = 0; k < wpo; ++k) chan_merge(tn, tm, tM, s_n[w + k], s_m[w + k], s_M[w + k]);
    const float var = tn > 0.f ? tM / tn : 0.f;  // biased
    mean[s] = tm;
    inv_std[s] = static_cast<float>(1.0 / sqrt(static_cast<double>(var) + static_cast<double>(eps)));
  }
}

int grid_for(long total, int block) {
  long g = (total + block - 1) / block;
  if (g < 1) g = 1;
  if (g > 65535L * 16) g = 65535L * 16;
  return static_cast<int>(g);
}

int vec_ec(int dtype, int C) {
  const int ec = dtype == 1 ? 8 : 4;
  return (C % ec == 0) ? ec : 1;
}

// ------------------------------------------------------------ streamed row walks
// The bandwidth-bound kernels below move NHWC rows through shared memory with
// bulk TMA copies (cp.async.bulk): a ring of kStreamStages chunks of R rows
// per input tensor, refilled by one thread, so that many bytes are in flight
// per SM without holding them in registers. One persistent block per SM walks
// a contiguous range of rows; every thread keeps a fixed group of EC channels.
constexpr int kStreamStages = 4;
constexpr int kChunkBytes = 16384;

template <int EC>
__device__ __forceinline__ void lds_v(const float* p, float (&v)[EC]) {
  const float4 t = *reinterpret_cast<const float4*>(p);
  v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
}
template <int EC>
__device__ __forceinline__ void lds_v(const __nv_bfloat16* p, float (&v)[EC]) {
  const uint4 t = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
    v[2 * e] = f.x;
    v[2 * e + 1] = f.y;
  }
}

// Elements e, e+1 of a per-thread channel group as one packed pair (f32x2 arithmetic below: the
// same operations as per element, two per instruction).
__device__ __forceinline__ float2 pr(const float* v, int e) { return make_float2(v[e], v[e + 1]); }
// act'(t) * dy (ReLU: a select, no multiply); FAST for layers stored in bf16 (see act_f)
template <int A, bool FAST>
__device__ __forceinline__ float dact_mul(float t, float dy) {
  if constexpr (A == 1) return t > 0.f ? dy : 0.f;
  else return dact_t<A, FAST>(t) * dy;
}

// The ReLU test on stored bf16 pre-activations, two channels per instruction and without forming t.
// t = gs * (v - mean) + beta > 0 (gs = gamma * inv_std) holds exactly when s * v > s * th, with
// th = mean - beta / gs and s the sign of gs. Because v is a bf16 value, s * v > s * th is the same as
// s * v > floor_bf16(s * th): a packed bf16 compare of v (sign bit flipped by an XOR where s < 0)
// with a key per channel, exact up to the fp32 rounding of th. gs == 0 leaves t = beta: a key of -inf
// (every v passes) or +inf (none does); a NaN gs gives a NaN key (none passes, as t would be NaN).
__device__ __forceinline__ void relu_key(float mean, float gs, float beta, uint32_t& key, uint32_t& sgn) {
  sgn = 0;
  if (gs > 0.f) {
    key = __bfloat16_as_ushort(__float2bfloat16_rd(mean - beta / gs));
  } else if (gs < 0.f) {
    key = __bfloat16_as_ushort(__float2bfloat16_rd(beta / gs - mean));
    sgn = 0x8000u;
  } else if (gs == 0.f) {
    key = beta > 0.f ? 0xff80u : 0x7f80u;
  } else {
    key = 0x7fc0u;
  }
}
// Keys of channels 2q and 2q+1 in the low and high halves of key[q] / sgn[q] (nmu = -mean).
template <int EC>
__device__ __forceinline__ void relu_keys(const float* nmu, const float* gs, const float* be, uint32_t* key,
                                          uint32_t* sgn) {
#pragma unroll
  for (int q = 0; q < EC / 2; ++q) {
    uint32_t k0, s0, k1, s1;
    relu_key(-nmu[2 * q], gs[2 * q], be[2 * q], k0, s0);
    relu_key(-nmu[2 * q + 1], gs[2 * q + 1], be[2 * q + 1], k1, s1);
    key[q] = k0 | (k1 << 16);
    sgn[q] = s0 | (s1 << 16);
  }
}
// 0xffff in each half of a packed bf16 pair v whose ReLU test passes, 0 elsewhere
__device__ __forceinline__ uint32_t relu_mask2(uint32_t v, uint32_t key, uint32_t sgn) {
  const uint32_t f = v ^ sgn;
  return __hgt2_mask(*reinterpret_cast<const __nv_bfloat162*>(&f), *reinterpret_cast<const __nv_bfloat162*>(&key));
}
// a packed bf16 pair as floats (low half first, as stored)
__device__ __forceinline__ float2 bf2f(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}
// Streamed backward kernels take the packed path for bf16 layers with no activation or ReLU.
template <typename T, int A>
constexpr bool kPackedBwd = std::is_same<T, __nv_bfloat16>::value && (A == 0 || A == 1);


__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Walk rows [r0, r1) of NIN tensors [rows][C] (EC channels per thread, the
// group g fixed per thread); proc(row, v) gets the NIN vectors of one row as floats, or with RAW
// proc(row, p) the NIN shared-memory addresses of the thread's EC elements, still in T.
// Returns false if a wait gave up (recorded in *err).
template <typename T, int EC, int NIN, bool RAW = false, typename Proc>
__device__ __forceinline__ bool stream_walk(const T* const (&in)[NIN], long r0, long r1, int C, int R, int g,
                                            int rl, int rpp, uint8_t* sm, uint64_t* full, int* err, int rev,
                                            Proc&& proc) {
  const size_t row_bytes = static_cast<size_t>(C) * sizeof(T);
  const uint32_t chunk = static_cast<uint32_t>(R * row_bytes);
  const long nchunks = r1 > r0 ? (r1 - r0 + R - 1) / R : 0;
  // first row of chunk k: forward from r0, or backward from r1 (the last chunk is the short one)
  auto chunk_begin = [&](long k) { return rev ? max(r0, r1 - (k + 1) * R) : r0 + k * R; };
  auto chunk_end = [&](long k) { return rev ? r1 - k * R : min(r1, r0 + (k + 1) * R); };
  auto issue = [&](long k) {
    const int s = static_cast<int>(k % kStreamStages);
    const long rb = chunk_begin(k);
    const long re = chunk_end(k);
    const uint32_t bytes = static_cast<uint32_t>((re - rb) * row_bytes);
    mbar_arrive_expect_tx(&full[s], NIN * bytes);
#pragma unroll
    for (int i = 0; i < NIN; ++i) bulk_load(smem_u32(sm + (s * NIN + i) * chunk), in[i] + rb * C, bytes, &full[s]);
  };
  if (threadIdx.x == 0)
    for (long k = 0; k < nchunks && k < kStreamStages; ++k) issue(k);
  bool ok = true;
  for (long k = 0; k < nchunks; ++k) {
    const int s = static_cast<int>(k % kStreamStages);
    const int w = wait(&full[s], static_cast<uint32_t>((k / kStreamStages) & 1), err, 7) ? 1 : 0;
    if (!__syncthreads_and(w)) {
      ok = false;
      break;
    }
    const long rb = chunk_begin(k);
    const int nrows = static_cast<int>(chunk_end(k) - rb);
    if (rl < rpp) {
      for (int rr = rl; rr < nrows; rr += rpp) {
        const T* src[NIN];
#pragma unroll
        for (int i = 0; i < NIN; ++i)
          src[i] = reinterpret_cast<const T*>(sm + (s * NIN + i) * chunk) + static_cast<size_t>(rr) * C + g * EC;
        if constexpr (RAW) {
          proc(rb + rr, src);
        } else {
          float v[NIN][EC];
#pragma unroll
          for (int i = 0; i < NIN; ++i) lds_v<EC>(src[i], v[i]);
          proc(rb + rr, v);
        }
      }
    }
    __syncthreads();  // stage s consumed by every thread
    if (threadIdx.x == 0 && k + kStreamStages < nchunks) issue(k + kStreamStages);
  }
  if (!ok && threadIdx.x == 0) {
    // let the copies already issued land before the block exits (each wait bounded)
    for (long k = 0; k < nchunks && k < kStreamStages; ++k) {
      const int s = static_cast<int>(k % kStreamStages);
      (void)mbar_try_wait(&full[s], 0);
    }
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 1000000ull) {
    }
  }
  return ok;
}

template <typename T, int EC, int NIN>
struct StreamSetup {
  int cg, tpr, rpp, rl, g, seg, lb;
  long r0, r1;
  __device__ StreamSetup(long seg_rows, int bps, int C, long rpb, int rev) {
    cg = C / EC;
    tpr = cg;  // the streamed path is used when C / EC <= kBlock
    rpp = kBlock / tpr;
    rl = threadIdx.x / tpr;
    g = threadIdx.x % tpr;
    const SegRange r = seg_range(seg_rows, bps, rpb, rev);
    seg = r.seg;
    lb = r.lb;
    r0 = r.r0;
    r1 = r.r1;
  }
};

__device__ __forceinline__ void stream_init(uint64_t* full) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStreamStages; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
}

template <typename T, int EC, int A>
__global__ void __launch_bounds__(kBlock, 1) bn_apply_stream(const T* __restrict__ pre, T* __restrict__ y,
                                                             long seg_rows, int bps, int C, long rpb, int R, int cpg,
                                                             int rev, const float* __restrict__ mean,
                                                             const float* __restrict__ inv_std,
                                                             const float* __restrict__ gamma,
                                                             const float* __restrict__ beta, int* err) {
  pdl_entry();
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t full[kStreamStages];
  stream_init(full);
  const StreamSetup<T, EC, 1> st(seg_rows, bps, C, rpb, rev);
  float nmu[EC], sc[EC], be[EC];
#pragma unroll
  for (int e = 0; e < EC; ++e) {
    const int c = st.g * EC + e;
    const int si = stat_index(cpg, st.seg, c, C);
    nmu[e] = -mean[si];
    sc[e] = gamma[c] * inv_std[si];
    be[e] = beta[c];
  }
  const T* const in[1] = {pre};
  {
    stream_walk<T, EC, 1>(in, st.r0, st.r1, C, R, st.g, st.rl, st.rpp, sm, full, err, rev,
                          [&](long row, const float (&v)[1][EC]) {
                            float o[EC];
#pragma unroll
                            for (int e = 0; e < EC; e += 2) {
                              // (x - mean) * gamma * inv_std + beta
                              const float2 t = __ffma2_rn(__fadd2_rn(pr(v[0], e), pr(nmu, e)), pr(sc, e), pr(be, e));
                              o[e] = act_t<A, kFastAct<T>>(t.x);
                              o[e + 1] = act_t<A, kFastAct<T>>(t.y);
                            }
                            store_v<EC>(y + row * C + st.g * EC, o);
                          });
  }
}

// part[b][c][3] = (rows, mean, M2) of channel c over the block's rows (streamed form of norm_stats_kernel)
template <typename T, int EC>
__global__ void __launch_bounds__(kBlock, 1) norm_stats_stream(const T* __restrict__ pre, long seg_rows, int bps,
                                                               int C, long rpb, int R, int rev,
                                                               float* __restrict__ part, int* err) {
  pdl_entry();
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t full[kStreamStages];
  __shared__ float s_n[kBlock], s_m[kBlock * EC], s_M[kBlock * EC];
  stream_init(full);
  const StreamSetup<T, EC, 1> st(seg_rows, bps, C, rpb, rev);
  float K[EC], s1[EC], s2[EC], nt = 0.f;
#pragma unroll
  for (int e = 0; e < EC; ++e) K[e] = s1[e] = s2[e] = 0.f;
  const T* const in[1] = {pre};
  stream_walk<T, EC, 1>(in, st.r0, st.r1, C, R, st.g, st.rl, st.rpp, sm, full, err, rev,
                        [&](long, const float (&v)[1][EC]) {
                          if (nt == 0.f) {
#pragma unroll
                            for (int e = 0; e < EC; ++e) K[e] = v[0][e];
                          }
#pragma unroll
                          for (int e = 0; e < EC; ++e) {
                            const float d = v[0][e] - K[e];
                            s1[e] += d;
                            s2[e] = fmaf(d, d, s2[e]);
                          }
                          nt += 1.f;
                        });
  s_n[threadIdx.x] = nt;
#pragma unroll
  for (int e = 0; e < EC; ++e) {
    s_m[threadIdx.x * EC + e] = nt > 0.f ? K[e] + s1[e] / nt : 0.f;
    s_M[threadIdx.x * EC + e] = nt > 0.f ? fmaxf(s2[e] - s1[e] * (s1[e] / nt), 0.f) : 0.f;
  }
  __syncthreads();
  if (st.rl == 0) {
    for (int e = 0; e < EC; ++e) {
      float n = 0.f, m = 0.f, M = 0.f;
      for (int k = 0; k < st.rpp; ++k) {
        const int t = k * st.tpr + st.g;
        const float nb = s_n[t];
        if (nb == 0.f) continue;
        const float nn = n + nb, d = s_m[t * EC + e] - m, f = nb / nn;
        m = fmaf(d, f, m);
        M += s_M[t * EC + e] + d * d * n * f;
        n = nn;
      }
      float* o = part + (static_cast<size_t>(st.lb) * C + st.g * EC + e) * 3;
      o[0] = n;
      o[1] = m;
      o[2] = M;
    }
  }
}

// part[b][c] = {sum d_norm, sum d_norm * z} (NV = 2), and with NV = 3 also sum (x - mean): with it the
// finalize forms dbias = sum d_conv without the d_conv pass (see sum_finalize_kernel, mode 2).
template <typename T, int EC, int A, int NV = 2>
__global__ void __launch_bounds__(kBlock, NV == 3 ? 2 : 3) bn_bwd_reduce_stream(const T* __restrict__ pre, const T* __restrict__ dy,
                                                                  long seg_rows, int bps, int C, long rpb, int R,
                                                                  int cpg, int rev, const float* __restrict__ mean,
                                                                  const float* __restrict__ inv_std,
                                                                  const float* __restrict__ gamma,
                                                                  const float* __restrict__ beta,
                                                                  float* __restrict__ part, int* err) {
  pdl_entry();
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t full[kStreamStages];
  stream_init(full);
  const StreamSetup<T, EC, 2> st(seg_rows, bps, C, rpb, rev);
  float nmu[EC], is[EC], ga[EC], be[EC], a[EC], b[EC], x3[EC];
#pragma unroll
  for (int e = 0; e < EC; ++e) {
    const int c = st.g * EC + e;
    const int si = stat_index(cpg, st.seg, c, C);
    nmu[e] = -mean[si];
    is[e] = inv_std[si];
    ga[e] = gamma[c];
    be[e] = beta[c];
    a[e] = b[e] = x3[e] = 0.f;
  }
  const T* const in[2] = {pre, dy};
  if constexpr (kPackedBwd<T, A>) {
    // b accumulates d_norm * (x - mean); the factor inv_std is applied once after the walk
    uint32_t key[EC / 2], sgn[EC / 2];
    if constexpr (A == 1) {
      float gs[EC];
#pragma unroll
      for (int e = 0; e < EC; ++e) gs[e] = ga[e] * is[e];
      relu_keys<EC>(nmu, gs, be, key, sgn);
    }
    stream_walk<T, EC, 2, true>(in, st.r0, st.r1, C, R, st.g, st.rl, st.rpp, sm, full, err, rev,
                                [&](long, const T* const (&p)[2]) {
                                  const uint4 pv = *reinterpret_cast<const uint4*>(p[0]);
                                  const uint4 pd = *reinterpret_cast<const uint4*>(p[1]);
                                  const uint32_t wv[4] = {pv.x, pv.y, pv.z, pv.w};
                                  const uint32_t wd[4] = {pd.x, pd.y, pd.z, pd.w};
#pragma unroll
                                  for (int q = 0; q < EC / 2; ++q) {
                                    const int e = 2 * q;
                                    const uint32_t m = A == 1 ? relu_mask2(wv[q], key[q], sgn[q]) : 0xffffffffu;
                                    const float2 dn = bf2f(wd[q] & m);
                                    const float2 d = __fadd2_rn(bf2f(wv[q]), pr(nmu, e));
                                    const float2 sa = __fadd2_rn(pr(a, e), dn);
                                    const float2 sb = __ffma2_rn(dn, d, pr(b, e));
                                    a[e] = sa.x;
                                    a[e + 1] = sa.y;
                                    b[e] = sb.x;
                                    b[e + 1] = sb.y;
                                    if constexpr (NV == 3) {
                                      const float2 s3 = __fadd2_rn(pr(x3, e), d);
                                      x3[e] = s3.x;
                                      x3[e + 1] = s3.y;
                                    }
                                  }
                                });
#pragma unroll
    for (int e = 0; e < EC; ++e) b[e] *= is[e];
  } else {
    stream_walk<T, EC, 2>(in, st.r0, st.r1, C, R, st.g, st.rl, st.rpp, sm, full, err, rev,
                          [&](long, const float (&v)[2][EC]) {
#pragma unroll
                            for (int e = 0; e < EC; e += 2) {
                              const float2 xm = __fadd2_rn(pr(v[0], e), pr(nmu, e));
                              const float2 z = __fmul2_rn(xm, pr(is, e));
                              const float2 t = __ffma2_rn(pr(ga, e), z, pr(be, e));
                              const float2 dn = make_float2(dact_mul<A, kFastAct<T>>(t.x, v[1][e]),
                                                            dact_mul<A, kFastAct<T>>(t.y, v[1][e + 1]));
                              const float2 sa = __fadd2_rn(pr(a, e), dn);
                              const float2 sb = __ffma2_rn(dn, z, pr(b, e));
                              a[e] = sa.x;
                              a[e + 1] = sa.y;
                              b[e] = sb.x;
                              b[e + 1] = sb.y;
                              if constexpr (NV == 3) {
                                const float2 s3 = __fadd2_rn(pr(x3, e), xm);
                                x3[e] = s3.x;
                                x3[e + 1] = s3.y;
                              }
                            }
                          });
  }
  // the ring is free once the walk has returned (every chunk consumed, or the copies of a walk that
  // gave up landed): it holds the block's per-thread sums (NV * kBlock * EC floats, at most 24 KB; make_walk's
  // chunks give a ring of two inputs at least 32 KB)
  __syncthreads();
  float* s_a = reinterpret_cast<float*>(sm);
  float* s_b = s_a + kBlock * EC;
  float* s_c = s_b + kBlock * EC;
#pragma unroll
  for (int e = 0; e < EC; ++e) {
    s_a[threadIdx.x * EC + e] = a[e];
    s_b[threadIdx.x * EC + e] = b[e];
    if constexpr (NV == 3) s_c[threadIdx.x * EC + e] = x3[e];
  }
  __syncthreads();
  if (st.rl == 0) {
    for (int e = 0; e < EC; ++e) {
      float sa = 0.f, sb = 0.f, sc = 0.f;
      for (int k = 0; k < st.rpp; ++k) {
        sa += s_a[(k * st.tpr + st.g) * EC + e];
        sb += s_b[(k * st.tpr + st.g) * EC + e];
        if constexpr (NV == 3) sc += s_c[(k * st.tpr + st.g) * EC + e];
      }
      float* o = part + (static_cast<size_t>(st.lb) * C + st.g * EC + e) * NV;
      o[0] = sa;
      o[1] = sb;
      if constexpr (NV == 3) o[2] = sc;
    }
  }
}

// d_conv (MODE 0: batch / layer norm, 1: no norm) and part[b][c] = sum d_conv.
// Without an activation three blocks fit an SM (registers capped for it); an activation needs more
// registers (ReLU on bf16: 87, and capped for three blocks it spills, which measured slower than two
// blocks without spills): two.
template <typename T, int EC, int MODE, int A>
__global__ void __launch_bounds__(kBlock, A == 0 ? 3 : 2) dconv_stream(const T* __restrict__ pre, const T* __restrict__ dy,
                                                          long seg_rows, int bps, int C, long rpb, int R, int cpg,
                                                          int rev, const float* __restrict__ mean,
                                                          const float* __restrict__ inv_std,
                                                          const float* __restrict__ gamma,
                                                          const float* __restrict__ beta,
                                                          const float* __restrict__ c12, T* __restrict__ dconv,
                                                          float* __restrict__ part, int* err) {
  pdl_entry();
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t full[kStreamStages];
  stream_init(full);
  const StreamSetup<T, EC, 2> st(seg_rows, bps, C, rpb, rev);
  float nmu[EC], is[EC], ga[EC], be[EC], nk1[EC], k2[EC], a[EC];
#pragma unroll
  for (int e = 0; e < EC; ++e) {
    const int c = st.g * EC + e;
    a[e] = 0.f;
    if (MODE == 0) {
      const int si = stat_index(cpg, st.seg, c, C);
      nmu[e] = -mean[si];
      is[e] = inv_std[si];
      ga[e] = gamma[c];
      be[e] = beta[c];
      float k1;
      norm_bwd_coef(c12, cpg, st.seg, c, C, ga[e], seg_rows, k1, k2[e]);
      nk1[e] = -k1;
    }
  }
  const T* const in[2] = {pre, dy};
  if constexpr (kPackedBwd<T, A>) {
    // MODE 0: d_conv = P * d_norm + (Q * (x - mean) + S), P = inv_std * gamma, Q = -inv_std^2 * k2,
    // S = -inv_std * k1 (the same terms as inv_std * (gamma * d_norm - k1 - z * k2), z = (x - mean) * inv_std);
    // MODE 1: d_conv = d_norm. The ReLU test has mean 0, gain 1 and beta 0 without a norm.
    uint32_t key[EC / 2], sgn[EC / 2];
    float P[EC], Q[EC], S[EC];
#pragma unroll
    for (int e = 0; e < EC; ++e) {
      if (MODE == 0) {
        P[e] = is[e] * ga[e];
        Q[e] = -is[e] * is[e] * k2[e];
        S[e] = is[e] * nk1[e];
      } else {
        nmu[e] = 0.f;
        P[e] = 1.f;
        be[e] = 0.f;
      }
    }
    if constexpr (A == 1) relu_keys<EC>(nmu, P, be, key, sgn);
    stream_walk<T, EC, 2, true>(in, st.r0, st.r1, C, R, st.g, st.rl, st.rpp, sm, full, err, rev,
                                [&](long row, const T* const (&p)[2]) {
                                  const uint4 pv = *reinterpret_cast<const uint4*>(p[0]);
                                  const uint4 pd = *reinterpret_cast<const uint4*>(p[1]);
                                  const uint32_t wv[4] = {pv.x, pv.y, pv.z, pv.w};
                                  const uint32_t wd[4] = {pd.x, pd.y, pd.z, pd.w};
                                  float o[EC];
#pragma unroll
                                  for (int q = 0; q < EC / 2; ++q) {
                                    const int e = 2 * q;
                                    const uint32_t m = A == 1 ? relu_mask2(wv[q], key[q], sgn[q]) : 0xffffffffu;
                                    const float2 dn = bf2f(wd[q] & m);
                                    float2 r = dn;
                                    if (MODE == 0) {
                                      const float2 d = __fadd2_rn(bf2f(wv[q]), pr(nmu, e));
                                      r = __ffma2_rn(pr(P, e), dn, __ffma2_rn(pr(Q, e), d, pr(S, e)));
                                    }
                                    o[e] = r.x;
                                    o[e + 1] = r.y;
                                    const float2 sa = __fadd2_rn(pr(a, e), r);
                                    a[e] = sa.x;
                                    a[e + 1] = sa.y;
                                  }
                                  store_v<EC>(dconv + row * C + st.g * EC, o);
                                });
  } else {
    stream_walk<T, EC, 2>(in, st.r0, st.r1, C, R, st.g, st.rl, st.rpp, sm, full, err, rev,
                          [&](long row, const float (&v)[2][EC]) {
                            float o[EC];
#pragma unroll
                            for (int e = 0; e < EC; e += 2) {
                              float2 r;
                              if (MODE == 0) {
                                // inv_std * (gamma * d_norm - k1 - z * k2)
                                const float2 z = __fmul2_rn(__fadd2_rn(pr(v[0], e), pr(nmu, e)), pr(is, e));
                                const float2 t = __ffma2_rn(pr(ga, e), z, pr(be, e));
                                const float2 dn =
                                    make_float2(dact_mul<A, kFastAct<T>>(t.x, v[1][e]),
                                                dact_mul<A, kFastAct<T>>(t.y, v[1][e + 1]));
                                const float2 u = __ffma2_rn(pr(ga, e), dn, pr(nk1, e));
                                r = __fmul2_rn(pr(is, e), __ffma2_rn(make_float2(-z.x, -z.y), pr(k2, e), u));
                              } else {
                                r = make_float2(dact_mul<A, kFastAct<T>>(v[0][e], v[1][e]),
                                                dact_mul<A, kFastAct<T>>(v[0][e + 1], v[1][e + 1]));
                              }
                              o[e] = r.x;
                              o[e + 1] = r.y;
                              const float2 sa = __fadd2_rn(pr(a, e), r);
                              a[e] = sa.x;
                              a[e + 1] = sa.y;
                            }
                            store_v<EC>(dconv + row * C + st.g * EC, o);
                          });
  }
  // the ring is free once the walk has returned: it holds the block's per-thread sums
  __syncthreads();
  float* s_a = reinterpret_cast<float*>(sm);
#pragma unroll
  for (int e = 0; e < EC; ++e) s_a[threadIdx.x * EC + e] = a[e];
  __syncthreads();
  if (st.rl == 0) {
    for (int e = 0; e < EC; ++e) {
      float sa = 0.f;
      for (int k = 0; k < st.rpp; ++k) sa += s_a[(k * st.tpr + st.g) * EC + e];
      part[static_cast<size_t>(st.lb) * C + st.g * EC + e] = sa;
    }
  }
}

}  // namespace

// Blocks per segment for a walk of `segs` segments with `resident` blocks
// resident on the GPU at once. Time model: waves * (rows per block + ovh),
// ovh standing for a block's start-up (barrier set-up, first copies) in rows;
// the smallest modelled time wins (ties go to fewer blocks).
static int pick_bps(int segs, long seg_rows, long resident, long ovh) {
  int best = 1;
  double best_t = 1e300;
  for (int b = 1; b <= 64; ++b) {
    const long rpb = (seg_rows + b - 1) / b;
    if (b > 1 && rpb < ovh / 2) break;
    const double waves = std::ceil(static_cast<double>(segs) * b / static_cast<double>(resident));
    const double t = waves * static_cast<double>(rpb + ovh);
    if (t < best_t * (1 - 1e-9)) {
      best_t = t;
      best = b;
    }
  }
  return best;
}

RowWalk make_walk(long rows, int C, int dtype, int sms, int segs, int cpg, int per_sm) {
  RowWalk w;
  w.rows = rows;
  w.C = C;
  w.cpg = cpg;
  w.err = nullptr;
  w.segs = segs < 1 ? 1 : segs;
  w.seg_rows = rows / w.segs;
  const int ec = vec_ec(dtype, C);
  const long row_bytes = static_cast<long>(C) * (dtype == 1 ? 2 : 4);
  w.stream = (ec > 1 && C / ec <= kBlock && row_bytes <= kChunkBytes) ? 1 : 0;
  const int cg = C / ec;
  const int tpr = cg < kBlock ? cg : kBlock;
  const int rpp = kBlock / tpr;
  // Streamed walks use half-size chunks so that two blocks of the two-input kernels fit on an SM
  // (their registers and shared memory allow two; per_sm blocks for a kernel that fits more, such as the
  // backward reduce): more warps to hide the latency of each chunk's arithmetic than one block per SM
  // with bigger chunks.
  long resident;
  if (w.stream) {
    w.R = static_cast<int>(std::max<long>(1, (kChunkBytes / 2) / row_bytes));
    if (w.R > rpp) w.R = w.R / rpp * rpp;  // whole passes of the block's rows per chunk
    resident = static_cast<long>(per_sm < 2 ? 2 : per_sm) * sms;
  } else {
    w.R = 0;
    resident = 8L * sms;
  }
  const long unit = std::max<long>(w.R, rpp);  // rows of one chunk (streamed) or one pass
  if (w.segs == 1) {
    // Several waves of blocks of about 28 units each, so that blocks finishing early on fast SMs
    // take more work (one wave of equal blocks waits for the slowest SM); at least one full wave, and a
    // whole number of waves (a last wave of a few blocks would run on a nearly idle GPU: the 256-image
    // 56 x 56 x 256 layer's backward reduce had 4.04 waves).
    long g = (rows + 28 * unit - 1) / (28 * unit);
    g = std::max<long>(1, (g + resident / 2) / resident) * resident;
    g = std::min(g, 8 * resident);
    g = std::min(g, (rows + unit - 1) / unit);  // no block without rows
    if (g < 1) g = 1;
    w.G = static_cast<int>(g);
    w.bps = w.G;
    w.rows_per_block = (rows + w.G - 1) / w.G;
    return w;
  }
  // several segments (one per image): blocks never straddle a segment and the last wave stays full
  w.bps = pick_bps(w.segs, w.seg_rows, resident, 2L * unit);
  w.G = w.segs * w.bps;
  w.rows_per_block = (w.seg_rows + w.bps - 1) / w.bps;
  return w;
}

#define DISPATCH_EC(dtype, C, FP32_CALL, BF16_CALL)                           \
  do {                                                                        \
    if ((dtype) == 1) {                                                       \
      if ((C) % 8 == 0) { constexpr int EC = 8; using T = __nv_bfloat16; BF16_CALL; } \
      else { constexpr int EC = 1; using T = __nv_bfloat16; BF16_CALL; }      \
    } else {                                                                  \
      if ((C) % 4 == 0) { constexpr int EC = 4; using T = float; FP32_CALL; } \
      else { constexpr int EC = 1; using T = float; FP32_CALL; }              \
    }                                                                         \
  } while (0)

cudaError_t launch_pack_channels(int dtype, const void* src, void* dst, long rows, int C, int Cp, cudaStream_t st) {
  const int g = grid_for(rows * Cp, 256);
  if (dtype == 1)
    launch_k(pack_channels_kernel<__nv_bfloat16>, g, 256, 0, st, 1, static_cast<const __nv_bfloat16*>(src),
                                                           static_cast<__nv_bfloat16*>(dst), rows, C, Cp);
  else
    launch_k(pack_channels_kernel<float>, g, 256, 0, st, 1, static_cast<const float*>(src), static_cast<float*>(dst), rows,
                                                   C, Cp);
  return cudaGetLastError();
}

cudaError_t launch_prep_fprop_weights(int dtype, const void* w, void* bhi, float* blo, int OC, int taps, int IC,
                                      int ICp, cudaStream_t st) {
  const int g = grid_for(static_cast<long>(OC) * taps * ICp, 256);
  if (dtype == 1)
    launch_k(prep_fprop_weights_kernel<__nv_bfloat16>, g, 256, 0, st, 1, static_cast<const __nv_bfloat16*>(w),
                                                                static_cast<__nv_bfloat16*>(bhi), nullptr, OC, taps,
                                                                IC, ICp);
  else
    launch_k(prep_fprop_weights_kernel<float>, g, 256, 0, st, 1, static_cast<const float*>(w), static_cast<float*>(bhi), blo,
                                                        OC, taps, IC, ICp);
  return cudaGetLastError();
}

cudaError_t launch_prep_dgrad_weights(int dtype, const void* w, void* bhi, float* blo, int OC, int KH, int KW,
                                      int IC, int ICp, int OCp, int S, int Kd, const DgradWeightTable& t,
                                      cudaStream_t st) {
  const int g = grid_for(static_cast<long>(ICp) * Kd, 256);
  if (dtype == 1)
    launch_k(prep_dgrad_weights_kernel<__nv_bfloat16>, g, 256, 0, st, 1, static_cast<const __nv_bfloat16*>(w),
                                                                static_cast<__nv_bfloat16*>(bhi), nullptr, OC, KH, KW,
                                                                IC, ICp, OCp, S, Kd, t);
  else
    launch_k(prep_dgrad_weights_kernel<float>, g, 256, 0, st, 1, static_cast<const float*>(w), static_cast<float*>(bhi), blo,
                                                        OC, KH, KW, IC, ICp, OCp, S, Kd, t);
  return cudaGetLastError();
}

cudaError_t launch_prep_dgrad_merged_weights(int dtype, const void* w, void* bhi, float* blo, int OC, int KH, int KW,
                                             int IC, int ICp, int OCp, int S, cudaStream_t st) {
  const int g = grid_for(static_cast<long>(ICp) * KH * KW * OCp, 256);
  if (dtype == 1)
    launch_k(prep_dgrad_merged_weights_kernel<__nv_bfloat16>, g, 256, 0, st, 1, static_cast<const __nv_bfloat16*>(w),
             static_cast<__nv_bfloat16*>(bhi), nullptr, OC, KH, KW, IC, ICp, OCp, S);
  else
    launch_k(prep_dgrad_merged_weights_kernel<float>, g, 256, 0, st, 1, static_cast<const float*>(w),
             static_cast<float*>(bhi), blo, OC, KH, KW, IC, ICp, OCp, S);
  return cudaGetLastError();
}

cudaError_t launch_bn_stats_finalize(const float* part, const RowWalk& wk, float eps, float momentum, float* mean,
                                     float* inv_std, float* rm, float* rv, cudaStream_t st) {
  launch_k(bn_stats_finalize_kernel, (wk.C + 3) / 4, 128, 0, st, 1, part, wk.G, wk.C, eps, momentum, mean, inv_std, rm, rv);
  return cudaGetLastError();
}

// Launch a streamed kernel: EC is 8 (bf16) or 4 (fp32); dynamic shared memory holds the chunk ring.
// STREAM_LAUNCH_ACT also makes the activation a compile-time constant A of the kernel, so that each
// activation gets its own register allocation (tanh and sigmoid need far more registers than ReLU).
#define STREAM_LAUNCH_ACT(act, dtype, NIN, KERNEL, ...)                         \
  do {                                                                          \
    switch (act) {                                                              \
      case 1: { constexpr int A = 1; STREAM_LAUNCH(dtype, NIN, KERNEL, __VA_ARGS__); } break; \
      case 2: { constexpr int A = 2; STREAM_LAUNCH(dtype, NIN, KERNEL, __VA_ARGS__); } break; \
      case 3: { constexpr int A = 3; STREAM_LAUNCH(dtype, NIN, KERNEL, __VA_ARGS__); } break; \
      default: { constexpr int A = 0; STREAM_LAUNCH(dtype, NIN, KERNEL, __VA_ARGS__); } break; \
    }                                                                           \
  } while (0)
#define STREAM_LAUNCH(dtype, NIN, KERNEL, ...)                                                           \
  do {                                                                                                  \
    const size_t es = (dtype) == 1 ? 2 : 4;                                                             \
    const size_t smem = static_cast<size_t>(kStreamStages) * (NIN) * wk.R * wk.C * es;                  \
    if ((dtype) == 1) {                                                                                 \
      constexpr int EC = 8;                                                                             \
      using T = __nv_bfloat16;                                                                          \
      cudaFuncSetAttribute(KERNEL, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)); \
      launch_k(KERNEL, wk.G, kBlock, smem, st, 1, __VA_ARGS__);                                                  \
    } else {                                                                                            \
      constexpr int EC = 4;                                                                             \
      using T = float;                                                                                  \
      cudaFuncSetAttribute(KERNEL, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)); \
      launch_k(KERNEL, wk.G, kBlock, smem, st, 1, __VA_ARGS__);                                                  \
    }                                                                                                   \
  } while (0)

// Walk arguments shared by every row-walk kernel: segment geometry and the layer-norm flag.
#define WALK_ARGS wk.seg_rows, wk.bps, wk.C, wk.rows_per_block
#define LN_FLAG wk.cpg

cudaError_t launch_bn_apply(int dtype, const void* pre, void* y, const RowWalk& wk, const float* mean,
                            const float* inv_std, const float* gamma, const float* beta, int act, int rev,
                            cudaStream_t st) {
  if (wk.stream) {
    STREAM_LAUNCH_ACT(act, dtype, 1, (bn_apply_stream<T, EC, A>), static_cast<const T*>(pre), static_cast<T*>(y),
                      WALK_ARGS, wk.R, LN_FLAG, rev, mean, inv_std, gamma, beta, wk.err);
    return cudaGetLastError();
  }
  DISPATCH_EC(dtype, wk.C,
              (launch_k(bn_apply_kernel<T, EC>, wk.G, kBlock, 0, st, 1, static_cast<const T*>(pre), static_cast<T*>(y),
                                                                 WALK_ARGS, LN_FLAG, mean, inv_std, gamma, beta,
                                                                 act)),
              (launch_k(bn_apply_kernel<T, EC>, wk.G, kBlock, 0, st, 1, static_cast<const T*>(pre), static_cast<T*>(y),
                                                                 WALK_ARGS, LN_FLAG, mean, inv_std, gamma, beta,
                                                                 act)));
  return cudaGetLastError();
}

cudaError_t launch_bn_bwd_reduce(int dtype, const void* pre, const void* dy, const RowWalk& wk, const float* mean,
                                 const float* inv_std, const float* gamma, const float* beta, int act, float* part,
                                 int nv, cudaStream_t st) {
  if (nv == 3) {
    // the third partial serves the backward that forms d_conv inside the GEMMs: streamed batch-norm walks
    // of bf16 layers with tanh or sigmoid only; two blocks per SM
    if (!(wk.stream && wk.cpg == 0 && dtype == 1 && (act == 2 || act == 3))) return cudaErrorInvalidValue;
    constexpr int EC = 8;
    using T = __nv_bfloat16;
    const size_t smem = static_cast<size_t>(kStreamStages) * 2 * wk.R * wk.C * sizeof(T);
    auto go = [&](auto kernel) {
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      launch_k(kernel, wk.G, kBlock, smem, st, 1, static_cast<const T*>(pre), static_cast<const T*>(dy), WALK_ARGS,
               wk.R, LN_FLAG, 0, mean, inv_std, gamma, beta, part, wk.err);
    };
    if (act == 2) go(bn_bwd_reduce_stream<T, EC, 2, 3>);
    else go(bn_bwd_reduce_stream<T, EC, 3, 3>);
    return cudaGetLastError();
  }
  if (wk.stream) {
    // three blocks per SM (registers capped for it); the column-sum scratch reuses the ring, so three
    // rings of full chunks fit in shared memory
    STREAM_LAUNCH_ACT(act, dtype, 2, (bn_bwd_reduce_stream<T, EC, A>), static_cast<const T*>(pre),
                      static_cast<const T*>(dy), WALK_ARGS, wk.R, LN_FLAG, 0, mean, inv_std, gamma, beta, part,
                      wk.err);
    return cudaGetLastError();
  }
  DISPATCH_EC(dtype, wk.C,
              (launch_k(bn_bwd_reduce_kernel<T, EC>, wk.G, kBlock, 0, st, 1, static_cast<const T*>(pre),
                                                                      static_cast<const T*>(dy), WALK_ARGS, LN_FLAG,
                                                                      mean, inv_std, gamma, beta, act, part)),
              (launch_k(bn_bwd_reduce_kernel<T, EC>, wk.G, kBlock, 0, st, 1, static_cast<const T*>(pre),
                                                                      static_cast<const T*>(dy), WALK_ARGS, LN_FLAG,
                                                                      mean, inv_std, gamma, beta, act, part)));
  return cudaGetLastError();
}

cudaError_t launch_sum_finalize(const float* part, const RowWalk& wk, int nv, int mode, float* c12, float* acc0,
                                float* acc1, cudaStream_t st) {
  launch_k(sum_finalize_kernel, wk.C, 128, 0, st, 1, part, wk.G, wk.C, nv, mode, c12, acc0, acc1);
  return cudaGetLastError();
}

cudaError_t launch_bn_bwd_fused_finalize(const float* part, const RowWalk& wk, const float* mean,
                                         const float* inv_std, const float* gamma, const float* beta, float* c12,
                                         float* dbeta, float* dgamma, float* dbias, float* tbl, cudaStream_t st) {
  launch_k(bn_bwd_fused_finalize_kernel, wk.C, 128, 0, st, 1, part, wk.G, wk.C, wk.rows, mean, inv_std, gamma, beta,
           c12, dbeta, dgamma, dbias, tbl);
  return cudaGetLastError();
}

cudaError_t launch_bn_bwd_apply(int dtype, const void* pre, const void* dy, const RowWalk& wk, int Cp,
                                const float* mean, const float* inv_std, const float* gamma, const float* beta,
                                int act, const float* c12, void* dconv, float* part, cudaStream_t st) {
  if (wk.stream && wk.C == Cp) {  // reversed: starts on the rows the backward reduce read last
    STREAM_LAUNCH_ACT(act, dtype, 2, (dconv_stream<T, EC, 0, A>), static_cast<const T*>(pre),
                      static_cast<const T*>(dy), WALK_ARGS, wk.R, LN_FLAG, 1, mean, inv_std, gamma, beta, c12,
                      static_cast<T*>(dconv), part, wk.err);
    return cudaGetLastError();
  }
  // the vector path needs C == Cp (EC divides C); otherwise one channel per thread
  DISPATCH_EC(dtype, (wk.C == Cp ? wk.C : 1),
              (launch_k(dconv_kernel<T, EC, 0>, wk.G, kBlock, 0, st, 1, static_cast<const T*>(pre),
                                                                 static_cast<const T*>(dy), wk.seg_rows, wk.bps, wk.C,
                                                                 Cp, wk.rows_per_block, LN_FLAG, mean, inv_std, gamma,
                                                                 beta, act, c12, static_cast<T*>(dconv), part)),
              (launch_k(dconv_kernel<T, EC, 0>, wk.G, kBlock, 0, st, 1, static_cast<const T*>(pre),
                                                                 static_cast<const T*>(dy), wk.seg_rows, wk.bps, wk.C,
                                                                 Cp, wk.rows_per_block, LN_FLAG, mean, inv_std, gamma,
                                                                 beta, act, c12, static_cast<T*>(dconv), part)));
  return cudaGetLastError();
}

cudaError_t launch_act_bwd(int dtype, const void* pre, const void* dy, const RowWalk& wk, int Cp, int act,
                           void* dconv, float* part, cudaStream_t st) {
  if (wk.stream && wk.C == Cp) {
    STREAM_LAUNCH_ACT(act, dtype, 2, (dconv_stream<T, EC, 1, A>), static_cast<const T*>(pre),
                      static_cast<const T*>(dy), WALK_ARGS, wk.R, 0, 1, nullptr, nullptr, nullptr, nullptr, nullptr,
                      static_cast<T*>(dconv), part, wk.err);
    return cudaGetLastError();
  }
  DISPATCH_EC(dtype, (wk.C == Cp ? wk.C : 1),
              (launch_k(dconv_kernel<T, EC, 1>, wk.G, kBlock, 0, st, 1, static_cast<const T*>(pre),
                                                                 static_cast<const T*>(dy), wk.seg_rows, wk.bps, wk.C,
                                                                 Cp, wk.rows_per_block, 0, nullptr, nullptr, nullptr,
                                                                 nullptr, act, nullptr, static_cast<T*>(dconv),
                                                                 part)),
              (launch_k(dconv_kernel<T, EC, 1>, wk.G, kBlock, 0, st, 1, static_cast<const T*>(pre),
                                                                 static_cast<const T*>(dy), wk.seg_rows, wk.bps, wk.C,
                                                                 Cp, wk.rows_per_block, 0, nullptr, nullptr, nullptr,
                                                                 nullptr, act, nullptr, static_cast<T*>(dconv),
                                                                 part)));
  return cudaGetLastError();
}

cudaError_t launch_ln_stats_finalize(const float* rstats, int n_images, long hw, int n_tiles, int halves, int BN,
                                     int hcols, int OC, float eps, float* mean, float* inv_std, cudaStream_t st) {
  launch_k(ln_stats_finalize_kernel, n_images, 256, 0, st, 1, rstats, n_tiles, halves, BN, hcols, OC, hw, eps, mean,
                                                     inv_std);
  return cudaGetLastError();
}

cudaError_t launch_norm_seg_finalize(const float* part, const RowWalk& wk, const float* gamma, float* out,
                                     cudaStream_t st) {
  const int n_out = wk.segs * (wk.C / wk.cpg);
  const int wpo = finalize_wpo(static_cast<long>(wk.bps) * wk.cpg), opb = 4 / wpo;
  launch_k(norm_seg_finalize_kernel, (n_out + opb - 1) / opb, 128, 0, st, 1, part, wk.bps, wk.C, wk.cpg, n_out, wpo, gamma,
                                                                     out);
  return cudaGetLastError();
}

cudaError_t launch_norm_stats(int dtype, const void* pre, const RowWalk& wk, int rev, float* part,
                              cudaStream_t st) {
  if (wk.stream) {
    STREAM_LAUNCH(dtype, 1, (norm_stats_stream<T, EC>), static_cast<const T*>(pre), WALK_ARGS, wk.R, rev, part,
                  wk.err);
    return cudaGetLastError();
  }
  DISPATCH_EC(dtype, wk.C,
              (launch_k(norm_stats_kernel<T, EC>, wk.G, kBlock, 0, st, 1, static_cast<const T*>(pre), WALK_ARGS, part)),
              (launch_k(norm_stats_kernel<T, EC>, wk.G, kBlock, 0, st, 1, static_cast<const T*>(pre), WALK_ARGS, part)));
  return cudaGetLastError();
}

cudaError_t launch_gn_stats_finalize(const float* part, const RowWalk& wk, float eps, float* mean, float* inv_std,
                                     cudaStream_t st) {
  const int n_out = wk.segs * (wk.C / wk.cpg);
  const int wpo = finalize_wpo(static_cast<long>(wk.bps) * wk.cpg), opb = 4 / wpo;
  launch_k(gn_stats_finalize_kernel, (n_out + opb - 1) / opb, 128, 0, st, 1, part, wk.bps, wk.C, wk.cpg, n_out, wpo, eps,
                                                                     mean, inv_std);
  return cudaGetLastError();
}

#undef WALK_ARGS
#undef LN_FLAG

cudaError_t launch_prep_col2im_weights(int dtype, const void* w, void* bhi, float* blo, int OC, int taps, int IC,
                                       int ICp, int OCp, cudaStream_t st) {
  const int g = grid_for(static_cast<long>(taps) * ICp * OCp, 256);
  if (dtype == 1)
    launch_k(prep_col2im_weights_kernel<__nv_bfloat16>, g, 256, 0, st, 1, static_cast<const __nv_bfloat16*>(w),
                                                                 static_cast<__nv_bfloat16*>(bhi), nullptr, OC, taps,
                                                                 IC, ICp, OCp);
  else
    launch_k(prep_col2im_weights_kernel<float>, g, 256, 0, st, 1, static_cast<const float*>(w), static_cast<float*>(bhi), blo,
                                                         OC, taps, IC, ICp, OCp);
  return cudaGetLastError();
}

cudaError_t launch_col2im(int dtype, const void* dcol, void* dx, int N, int H, int W, int IC, int ICp, int OH, int OW,
                          int KH, int KW, int S, int P, cudaStream_t st) {
  DISPATCH_EC(dtype, IC,
              (launch_k(col2im_kernel<T, EC>, grid_for(static_cast<long>(N) * H * W * (IC / EC), 256), 256, 0, st, 1,
                  static_cast<const T*>(dcol), static_cast<T*>(dx), N, H, W, IC, ICp, OH, OW, KH, KW, S, P)),
              (launch_k(col2im_kernel<T, EC>, grid_for(static_cast<long>(N) * H * W * (IC / EC), 256), 256, 0, st, 1,
                  static_cast<const T*>(dcol), static_cast<T*>(dx), N, H, W, IC, ICp, OH, OW, KH, KW, S, P)));
  return cudaGetLastError();
}

cudaError_t launch_wgrad_reduce(const float* partial, int splits, int OC, int taps, int ICp, int IC, float* dw,
                                const float* bpart, int bG, float* dbias, cudaStream_t st) {
  const int nbias = dbias ? OC : 0;  // one more block per channel for the dbias sums
  // Few splits: one thread per item over every split (measured faster for the 25 splits of a 256-image
  // 3 x 3 layer). Many splits (the fp32 layers, 1 x 1 layers with one row tile): the split groups, which
  // shorten each thread's chain of dependent loads.
  if (splits < kRedSerialMax) {
    const int V = (IC == ICp && IC % 4 == 0) ? 4 : 1;  // channels per thread (see the kernel)
    const int g = grid_for(static_cast<long>(OC) * taps * IC / V, 256);
    launch_k(wgrad_reduce_serial_kernel, g + nbias, 256, 0, st, 1, partial, splits, OC, taps, ICp, IC, dw, g, bpart,
             bG, dbias);
    return cudaGetLastError();
  }
  // 32 items of V channels per block (see the kernel)
  if (IC == ICp && IC % 4 == 0) {
    const int g = static_cast<int>((static_cast<long>(OC) * taps * IC / 4 + 31) / 32);
    launch_k(wgrad_reduce_kernel<4>, g + nbias, 32 * kRedGroups, 0, st, 1, partial, splits, OC, taps, ICp, IC, dw, g,
             bpart, bG, dbias);
  } else {
    const int g = static_cast<int>((static_cast<long>(OC) * taps * IC + 31) / 32);
    launch_k(wgrad_reduce_kernel<1>, g + nbias, 32 * kRedGroups, 0, st, 1, partial, splits, OC, taps, ICp, IC, dw, g,
             bpart, bG, dbias);
  }
  return cudaGetLastError();
}

cudaError_t launch_bn_eval_stats(const float* rm, const float* rv, float eps, int C, float* mean, float* inv_std,
                                 cudaStream_t st) {
  launch_k(bn_eval_stats_kernel, (C + 127) / 128, 128, 0, st, 1, rm, rv, eps, C, mean, inv_std);
  return cudaGetLastError();
}

cudaError_t launch_infer_fold(const float* bias, const float* gamma, const float* beta, const float* rm,
                              const float* rv, float eps, int norm, int OC, float* scale, float* shift,
                              cudaStream_t st) {
  launch_k(infer_fold_kernel, (OC + 127) / 128, 128, 0, st, 1, bias, gamma, beta, rm, rv, eps, norm, OC, scale, shift);
  return cudaGetLastError();
}

}  // namespace c2d
