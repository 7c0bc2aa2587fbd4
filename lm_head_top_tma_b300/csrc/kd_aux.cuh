// SIMT kernels around the tensor-core GEMMs of the chunk loop:
//   prep     teacher-cache rows -> ids sorted ascending (with their p), the
//            teacher mass M_t = sum_k p_tk and E_t = sum_k p_tk log p_tk,
//            plus the id range check;
//   combine  per-(row, vocabulary tile) softmax partials -> lse_t and the
//            per-row loss L_t = E_t - sum_k p_tk z_tk + M_t lse_t;
//   reductions of the loss (fp64, fixed order) and of split-K dH partials;
//   g_from_e the gradient operand G = M_t softmax(z_t) - p at the ids, formed
//            in place from the exponentials the forward GEMM kept (the fused
//            step without the backward recompute).
#pragma once

#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "kd_ptx.cuh"
#include "kdtopk.h"

namespace kd {

constexpr int PREP_WARPS = 4;

// One warp per chunk row.  The row's K (id, p) pairs are held in registers,
// EPT = Kpad / 32 consecutive slots per lane (Kpad: the power of two >= K,
// padding ids INT_MAX), loaded 16 bytes at a time when the row allows it, and
// sorted ascending by id with a bitonic network: exchanges across lanes by
// shuffles, within a lane by register swaps.  Equal ids keep their pairs
// (neither partner takes the other's), so duplicates survive intact.
template <int EPT>
__global__ void __launch_bounds__(PREP_WARPS * 32)
    kd_prep_kernel(const int32_t* __restrict__ idx, const float* __restrict__ p, int rows_valid,
                   int Cpad, int K, int V, int vec_rows, int32_t* __restrict__ sidx, float* __restrict__ sp,
                   float* __restrict__ rowM, float* __restrict__ rowE, int* status) {
  constexpr int N = 32 * EPT;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * PREP_WARPS + warp;
  if (r >= Cpad) return;
  const bool live = r < rows_valid;
  const int e0 = lane * EPT;  // this lane's first slot
  int key[EPT];
  float val[EPT];
#pragma unroll
  for (int i = 0; i < EPT; ++i) {
    key[i] = INT_MAX;
    val[i] = 0.f;
  }
  bool bad = false;
  if (live) {
    const int32_t* ir = idx + static_cast<size_t>(r) * K;
    const float* pr = p + static_cast<size_t>(r) * K;
    if constexpr (EPT >= 4) {
      if (vec_rows) {  // K % 4 == 0 and 16-byte aligned rows
#pragma unroll
        for (int i = 0; i < EPT; i += 4) {
          if (e0 + i < K) {  // K % 4 == 0: the whole 4-slot group is valid
            const int4 a = __ldg(reinterpret_cast<const int4*>(ir + e0 + i));
            const float4 b = __ldg(reinterpret_cast<const float4*>(pr + e0 + i));
            key[i] = a.x;
            key[i + 1] = a.y;
            key[i + 2] = a.z;
            key[i + 3] = a.w;
            val[i] = b.x;
            val[i + 1] = b.y;
            val[i + 2] = b.z;
            val[i + 3] = b.w;
          }
        }
      }
    }
    if (!(EPT >= 4 && vec_rows)) {
#pragma unroll
      for (int i = 0; i < EPT; ++i)
        if (e0 + i < K) {
          key[i] = __ldg(ir + e0 + i);
          val[i] = __ldg(pr + e0 + i);
        }
    }
#pragma unroll
    for (int i = 0; i < EPT; ++i)
      if (e0 + i < K && (key[i] < 0 || key[i] >= V)) bad = true;
  }
  bad = __any_sync(0xffffffffu, bad);

#pragma unroll
  for (int size = 2; size <= N; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= EPT) {  // partner slot in lane ^ (stride / EPT), same position
        const int lm = stride / EPT;
        const bool lower = (lane & lm) == 0;
#pragma unroll
        for (int i = 0; i < EPT; ++i) {
          const bool up = ((e0 + i) & size) == 0;
          const int k2 = __shfl_xor_sync(0xffffffffu, key[i], lm);
          const float v2 = __shfl_xor_sync(0xffffffffu, val[i], lm);
          const bool take = (lower == up) ? (k2 < key[i]) : (k2 > key[i]);
          if (take) {
            key[i] = k2;
            val[i] = v2;
          }
        }
      } else {  // both slots in this lane
#pragma unroll
        for (int i = 0; i < EPT; ++i) {
          if ((i & stride) == 0) {
            const int j = i | stride;
            const bool up = ((e0 + i) & size) == 0;
            if ((key[i] > key[j]) == up) {
              const int tk = key[i];
              key[i] = key[j];
              key[j] = tk;
              const float tv = val[i];
              val[i] = val[j];
              val[j] = tv;
            }
          }
        }
      }
    }
  }

  float m = 0.f, e = 0.f;
#pragma unroll
  for (int i = 0; i < EPT; ++i) {
    m += val[i];
    if (val[i] > 0.f) e += val[i] * logf(val[i]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    m += __shfl_xor_sync(0xffffffffu, m, o);
    e += __shfl_xor_sync(0xffffffffu, e, o);
  }
  if (bad) {  // the row contributes nothing; the caller learns it from the status word
    m = 0.f;
    e = 0.f;
#pragma unroll
    for (int i = 0; i < EPT; ++i) {
      key[i] = INT_MAX;
      val[i] = 0.f;
    }
  }
  int32_t* so = sidx + static_cast<size_t>(r) * K;
  float* po = sp + static_cast<size_t>(r) * K;
  if constexpr (EPT >= 4) {
    if (vec_rows) {
#pragma unroll
      for (int i = 0; i < EPT; i += 4) {
        if (e0 + i < K) {
          *reinterpret_cast<int4*>(so + e0 + i) = make_int4(key[i], key[i + 1], key[i + 2], key[i + 3]);
          *reinterpret_cast<float4*>(po + e0 + i) = make_float4(val[i], val[i + 1], val[i + 2], val[i + 3]);
        }
      }
    }
  }
  if (!(EPT >= 4 && vec_rows)) {
#pragma unroll
    for (int i = 0; i < EPT; ++i)
      if (e0 + i < K) {
        so[e0 + i] = key[i];
        po[e0 + i] = val[i];
      }
  }
  if (lane == 0) {
    rowM[r] = m;
    rowE[r] = e;
    if (bad) atomicCAS(status, 0, KD_ERR_BAD_INDEX);
  }
}

constexpr int COMBINE_WARPS = 32;

// Block = 32 rows x 32 warps; warp w folds vocabulary tiles w, w+32, ...
// (four loads in flight per thread), warp 0 folds the 32 warp results.
__global__ void __launch_bounds__(COMBINE_WARPS * 32)
    kd_combine_kernel(const float* __restrict__ pm, const float* __restrict__ ps,
                      const float* __restrict__ ppz, int nt, int ld_part, int rows_valid,
                      const float* __restrict__ rowM, const float* __restrict__ rowE,
                      float* __restrict__ lse_out, float* __restrict__ loss_rows_out,
                      double* __restrict__ Lrow) {
  __shared__ float s_m[COMBINE_WARPS][32], s_s[COMBINE_WARPS][32], s_z[COMBINE_WARPS][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x * 32 + lane;
  float m = -INFINITY, s = 0.f, z = 0.f;
  if (r < rows_valid) {
    constexpr int U = 4;
    for (int t0 = warp; t0 < nt; t0 += COMBINE_WARPS * U) {
      float a[U], b[U], c[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int t = t0 + u * COMBINE_WARPS;
        const size_t o = static_cast<size_t>(t) * ld_part + r;
        a[u] = t < nt ? pm[o] : -INFINITY;
        b[u] = t < nt ? ps[o] : 0.f;
        c[u] = t < nt ? ppz[o] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        z += c[u];
        if (a[u] > m) {
          s = s * ex2(m - a[u]) + b[u];
          m = a[u];
        } else if (a[u] > -INFINITY) {
          s += b[u] * ex2(a[u] - m);
        }
      }
    }
  }
  s_m[warp][lane] = m;
  s_s[warp][lane] = s;
  s_z[warp][lane] = z;
  __syncthreads();
  if (warp == 0 && r < rows_valid) {
    float M2 = -INFINITY, S = 0.f, Z = 0.f;
    for (int w = 0; w < COMBINE_WARPS; ++w) {
      const float a = s_m[w][lane], b = s_s[w][lane];
      Z += s_z[w][lane];
      if (a > M2) {
        S = S * ex2(M2 - a) + b;
        M2 = a;
      } else if (a > -INFINITY) {
        S += b * ex2(a - M2);
      }
    }
    const float lse = (M2 + log2f(S)) * kLn2;
    const double L = static_cast<double>(rowE[r]) - static_cast<double>(Z) +
                     static_cast<double>(rowM[r]) * static_cast<double>(lse);
    lse_out[r] = lse;
    if (loss_rows_out) loss_rows_out[r] = static_cast<float>(L);
    Lrow[r] = L;
  }
}

// acc = (first ? 0 : acc) + sum of Lrow[0..rows) in a fixed order; on the
// last chunk also writes the fp32 loss.
__global__ void __launch_bounds__(1024)
    kd_loss_reduce_kernel(const double* __restrict__ Lrow, int rows, double* acc, int first,
                          float* loss_out) {
  __shared__ double sm[1024];
  double s = 0.0;
  for (int i = threadIdx.x; i < rows; i += 1024) s += Lrow[i];
  sm[threadIdx.x] = s;
  __syncthreads();
  for (int w = 512; w > 0; w >>= 1) {
    if (threadIdx.x < w) sm[threadIdx.x] += sm[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double tot = (first ? 0.0 : *acc) + sm[0];
    *acc = tot;
    if (loss_out) *loss_out = static_cast<float>(tot);
  }
}

// dH[r, :] = scale * sum_s part[s, r, :] for the chunk's valid rows.
__global__ void kd_dh_reduce_kernel(const float4* __restrict__ part, int S, int64_t split_stride4,
                                    int64_t n4, float scale, float4* __restrict__ dH) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float4 a = part[i];
    for (int s = 1; s < S; ++s) {
      const float4 b = part[s * split_stride4 + i];
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
    a.x *= scale;
    a.y *= scale;
    a.z *= scale;
    a.w *= scale;
    dH[i] = a;
  }
}

// dst[i] = bf16(scale * src[i]) (round to nearest even), 4 elements per thread
// when both pointers allow 16-/8-byte accesses.
__global__ void kd_scale_to_bf16_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst, int64_t n,
                                        float scale) {
  const int64_t n4 = n / 4;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 v = reinterpret_cast<const float4*>(src)[i];
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x * scale, v.y * scale);
    __nv_bfloat162 b = __floats2bfloat162_rn(v.z * scale, v.w * scale);
    uint2 w;
    w.x = *reinterpret_cast<uint32_t*>(&a);
    w.y = *reinterpret_cast<uint32_t*>(&b);
    reinterpret_cast<uint2*>(dst)[i] = w;
  }
  for (int64_t i = n4 * 4 + blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    dst[i] = __float2bfloat16_rn(src[i] * scale);
}

constexpr int GPASS_THREADS = 256;
constexpr int GPASS_VEC = 8;     // bf16 per 16-byte access
constexpr int GPASS_UNROLL = 4;  // accesses in flight per thread
constexpr int GPASS_TILE = 256;  // vocabulary tile of the partials
constexpr int GPASS_MAXK = 1024;

// In place over the rows of the chunk's operand buffer:
//   G[r, j] = bf16( M_r * e[r, j] * 2^(m[r, j / 256] - lse_r log2 e) - sum_{k: id_rk = j} p_rk )
// where e = 2^(z log2 e - m) was rounded to bf16 by the forward GEMM and m is
// that tile's base-2 row maximum (the softmax partials).  The teacher
// correction is subtracted in fp32 before the single rounding.  Columns in
// [V, ldg) are set to 0.  One block per row (rows r = blockIdx.x, + gridDim.x,
// ...): thread t visits 16-byte groups t, t + 256, ... in increasing column
// order, so a per-thread cursor over the row's sorted ids (staged in shared
// memory) finds the corrections of each group.
__global__ void __launch_bounds__(GPASS_THREADS)
    kd_g_from_e_kernel(__nv_bfloat16* __restrict__ G, int64_t ldg, int rows, int V, int K,
                       const int32_t* __restrict__ sidx, const float* __restrict__ sp,
                       const float* __restrict__ rowM, const float* __restrict__ lse,
                       const float* __restrict__ part_m, int ld_part) {
  __shared__ int s_id[GPASS_MAXK + 1];
  __shared__ float s_p[GPASS_MAXK];
  const int ngroups = static_cast<int>(ldg / GPASS_VEC);
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    __syncthreads();  // the previous row's ids are no longer read
    for (int k = threadIdx.x; k < K; k += GPASS_THREADS) {
      s_id[k] = __ldg(sidx + static_cast<size_t>(r) * K + k);
      s_p[k] = __ldg(sp + static_cast<size_t>(r) * K + k);
    }
    if (threadIdx.x == 0) s_id[K] = INT_MAX;  // sentinel
    __syncthreads();
    const float Mr = __ldg(rowM + r);
    const float nl2 = -__ldg(lse + r) * kLog2e;
    const float* pmr = part_m + r;
    __nv_bfloat16* grow = G + static_cast<size_t>(r) * ldg;
    int cur = 0;  // first sorted id not below this thread's next group
    for (int g0 = threadIdx.x; g0 < ngroups; g0 += GPASS_THREADS * GPASS_UNROLL) {
      uint4 raw[GPASS_UNROLL];
      float scale[GPASS_UNROLL];
#pragma unroll
      for (int u = 0; u < GPASS_UNROLL; ++u) {
        const int g = g0 + u * GPASS_THREADS;
        if (g < ngroups) {
          raw[u] = *reinterpret_cast<const uint4*>(grow + static_cast<size_t>(g) * GPASS_VEC);
          scale[u] = __ldg(pmr + static_cast<size_t>(g * GPASS_VEC / GPASS_TILE) * ld_part);
        }
      }
#pragma unroll
      for (int u = 0; u < GPASS_UNROLL; ++u) {
        const int g = g0 + u * GPASS_THREADS;
        if (g >= ngroups) break;
        const int col = g * GPASS_VEC;
        const float sc = Mr * ex2(scale[u] + nl2);
        const __nv_bfloat162* e2 = reinterpret_cast<const __nv_bfloat162*>(&raw[u]);
        float v[GPASS_VEC];
#pragma unroll
        for (int j = 0; j < GPASS_VEC / 2; ++j) {
          const float2 f = __bfloat1622float2(e2[j]);
          v[2 * j] = f.x * sc;
          v[2 * j + 1] = f.y * sc;
        }
        while (s_id[cur] < col) ++cur;
        for (int k = cur; s_id[k] < col + GPASS_VEC; ++k) {
          const int off = s_id[k] - col;
          const float pv = s_p[k];
#pragma unroll
          for (int j = 0; j < GPASS_VEC; ++j) v[j] = (j == off) ? v[j] - pv : v[j];
        }
#pragma unroll
        for (int j = 0; j < GPASS_VEC; ++j)
          if (col + j >= V) v[j] = 0.f;
        uint4 outv;
        __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&outv);
#pragma unroll
        for (int j = 0; j < GPASS_VEC / 2; ++j) o2[j] = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
        *reinterpret_cast<uint4*>(grow + col) = outv;
      }
    }
  }
}

}  // namespace kd
