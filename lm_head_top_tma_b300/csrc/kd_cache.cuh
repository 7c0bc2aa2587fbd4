// Offline teacher-cache builder: for each row of teacher logits Z[T, V] the K
// largest logits' ids (largest first, equal logits by ascending id) and their
// softmax probabilities p = exp(z - lse) (so the row's mass M_t = sum_k p <= 1).
// This is the "keep the top-100 of every token" step of the pipeline the pages
// describe (thorstenmeyerai.com, pipeline steps "Infer once" / "Select top-K";
// aimodeling.com "First cut": top-100 probabilities cached for every token),
// here over logits that are already on the device.
//
// One block of 1024 threads per row (grid-stride over rows); the row is read
// from HBM once and a second time from L2:
//   pass 1  per-thread maximum key and online (max, sum of 2^x) for lse;
//   select  theta = the K-th largest of the 1024 per-thread maxima: at least K
//           distinct elements reach it, so every top-K element has key >= theta;
//   pass 2  collect the elements with key >= theta (typically a few hundred)
//           into shared memory and sort them by (key descending, id ascending);
//   fallback  when more than CACHE_CAP elements reach theta (heavily tied or
//           adversarial rows) the exact K-th key is found by a binary search
//           over the key space, and the tied elements at it are taken in
//           ascending id order by an ordered block scan.
// Keys are the order-preserving unsigned images of the logits (sign bit
// flipped for positives, all bits for negatives), so comparisons are exact.
#pragma once

#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "kd_ptx.cuh"
#include "kdtopk.h"

namespace kd {

constexpr int CACHE_THREADS = 1024;
constexpr int CACHE_CAP = 4096;  // candidates kept in shared memory

template <typename T>
struct LogitTraits;

template <>
struct LogitTraits<float> {
  using Key = uint32_t;
  static constexpr int KEY_BITS = 32;
  __device__ static float value(float x) { return x; }
  __device__ static uint32_t key(float x) {
    const uint32_t b = __float_as_uint(x);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  }
};

template <>
struct LogitTraits<__nv_bfloat16> {
  using Key = uint32_t;  // 16 significant bits
  static constexpr int KEY_BITS = 16;
  __device__ static float value(__nv_bfloat16 x) { return __bfloat162float(x); }
  __device__ static uint32_t key(__nv_bfloat16 x) {
    const uint32_t b = static_cast<uint32_t>(__bfloat16_as_ushort(x));
    return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
  }
};

// Sorts n_pad (a power of two) 64-bit composite keys ascending in shared
// memory; all threads of the block call it.
__device__ __forceinline__ void block_bitonic_sort_u64(uint64_t* a, int n_pad) {
  for (int size = 2; size <= n_pad; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n_pad; i += blockDim.x) {
        const int j = i ^ stride;
        if (j > i) {
          const bool up = (i & size) == 0;
          const uint64_t x = a[i], y = a[j];
          if ((x > y) == up) {
            a[i] = y;
            a[j] = x;
          }
        }
      }
      __syncthreads();
    }
  }
}

// Block-wide sum of an int (all threads call; result valid in every thread).
__device__ __forceinline__ int block_sum_int(int v, int* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int t = lane < static_cast<int>(blockDim.x >> 5) ? red[lane] : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
  return t;
}

template <typename TL>
__global__ void __launch_bounds__(CACHE_THREADS)
    kd_topk_cache_kernel(const TL* __restrict__ Z, int64_t T, int V, int K, int32_t* __restrict__ idx_out,
                         float* __restrict__ p_out, float* __restrict__ lse_out) {
  using Tr = LogitTraits<TL>;
  __shared__ uint64_t cand[CACHE_CAP];  // (~key << 32) | id: ascending = key descending, id ascending
  __shared__ float red_m[32], red_s[32];
  __shared__ int red_i[32];
  __shared__ int s_count;
  __shared__ float s_lse;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  constexpr int NW = CACHE_THREADS / 32;

  for (int64_t row = blockIdx.x; row < T; row += gridDim.x) {
    const TL* z = Z + row * static_cast<int64_t>(V);
    // ---------------- pass 1: per-thread max key, online softmax normaliser
    uint32_t kmax = 0;
    float m = -INFINITY, s = 0.f;
    for (int j = tid; j < V; j += CACHE_THREADS) {
      const TL x = z[j];
      const float v = Tr::value(x) * kLog2e;
      kmax = max(kmax, Tr::key(x));
      if (v > m) {
        s = s * ex2(m - v) + 1.f;
        m = v;
      } else if (v > -INFINITY) {  // masked (-inf) logits carry no probability
        s += ex2(v - m);
      }
    }
    // block (max, sum) in base 2
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
      const float mn = fmaxf(m, m2);
      s = (mn == -INFINITY) ? 0.f : s * ex2(m - mn) + s2 * ex2(m2 - mn);
      m = mn;
    }
    __syncthreads();  // the previous row's shared state is no longer read
    if (lane == 0) {
      red_m[warp] = m;
      red_s[warp] = s;
    }
    // the K-th largest per-thread maximum: sort the 1024 maxima (descending via ~key)
    cand[tid] = (static_cast<uint64_t>(~kmax) << 32) | static_cast<uint32_t>(tid);
    __syncthreads();
    if (warp == 0) {
      float mm = lane < NW ? red_m[lane] : -INFINITY;
      float ss = lane < NW ? red_s[lane] : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, mm, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, ss, o);
        const float mn = fmaxf(mm, m2);
        ss = (mn == -INFINITY) ? 0.f : ss * ex2(mm - mn) + s2 * ex2(m2 - mn);
        mm = mn;
      }
      if (lane == 0) s_lse = (mm + log2f(ss)) * kLn2;
    }
    block_bitonic_sort_u64(cand, CACHE_THREADS);
    // threads beyond V contributed kmax = 0, the smallest key; theta <= the K-th largest element's key
    const uint32_t theta = ~static_cast<uint32_t>(cand[K - 1] >> 32);
    if (tid == 0) s_count = 0;
    __syncthreads();

    // ---------------- pass 2: candidates with key >= theta
    for (int j = tid; j < V; j += CACHE_THREADS) {
      const uint32_t k = Tr::key(z[j]);
      if (k >= theta) {
        const int at = atomicAdd(&s_count, 1);
        if (at < CACHE_CAP) cand[at] = (static_cast<uint64_t>(~k) << 32) | static_cast<uint32_t>(j);
      }
    }
    __syncthreads();
    int n = s_count;
    if (n > CACHE_CAP) {
      // ---------------- fallback: exact K-th key by binary search, then ordered ties
      // largest kappa with count(key >= kappa) >= K, searched in [theta, 2^bits - 1]
      uint64_t lo = theta, hi = (Tr::KEY_BITS == 32) ? 0xFFFFFFFFull : 0xFFFFull;
      while (lo < hi) {
        const uint64_t mid = lo + (hi - lo + 1) / 2;
        int c = 0;
        for (int j = tid; j < V; j += CACHE_THREADS) c += static_cast<uint64_t>(Tr::key(z[j])) >= mid;
        if (block_sum_int(c, red_i) >= K) lo = mid;
        else hi = mid - 1;
      }
      const uint32_t kappa = static_cast<uint32_t>(lo);
      __syncthreads();
      if (tid == 0) s_count = 0;
      __syncthreads();
      for (int j = tid; j < V; j += CACHE_THREADS) {  // fewer than K are strictly above kappa
        const uint32_t k = Tr::key(z[j]);
        if (k > kappa) cand[atomicAdd(&s_count, 1)] = (static_cast<uint64_t>(~k) << 32) | static_cast<uint32_t>(j);
      }
      __syncthreads();
      int taken = s_count;
      // ties at kappa in ascending id order, one block-wide segment at a time
      for (int base = 0; base < V && taken < K; base += CACHE_THREADS) {
        const int j = base + tid;
        const bool tie = j < V && Tr::key(z[j]) == kappa;
        const unsigned bal = __ballot_sync(0xffffffffu, tie);
        __syncthreads();
        if (lane == 0) red_i[warp] = __popc(bal);
        __syncthreads();
        int before = 0;
        for (int w = 0; w < warp; ++w) before += red_i[w];
        const int rank_in = before + __popc(bal & ((1u << lane) - 1u));
        if (tie && taken + rank_in < K)
          cand[taken + rank_in] = (static_cast<uint64_t>(~kappa) << 32) | static_cast<uint32_t>(j);
        int total = 0;
        for (int w = 0; w < NW; ++w) total += red_i[w];
        taken += total;
      }
      n = K;
      __syncthreads();
    }
    // ---------------- sort the candidates and emit the top K
    int n_pad = 1;
    while (n_pad < n) n_pad <<= 1;
    for (int i = n + tid; i < n_pad; i += CACHE_THREADS) cand[i] = ~0ull;
    __syncthreads();
    block_bitonic_sort_u64(cand, n_pad);
    const float lse = s_lse;
    for (int k = tid; k < K; k += CACHE_THREADS) {
      const int id = static_cast<int>(cand[k] & 0xFFFFFFFFu);
      idx_out[row * K + k] = id;
      p_out[row * K + k] = ex2((Tr::value(z[id]) - lse) * kLog2e);
    }
    if (tid == 0 && lse_out) lse_out[row] = lse;
  }
}

}  // namespace kd
