// Offline teacher-cache builder: for each row of teacher logits Z[T, V] the K
// largest logits' ids (largest first, equal logits by ascending id) and their
// softmax probabilities p = exp(z - lse) (so the row's mass M_t = sum_k p <= 1).
// This is the "keep the top-100 of every token" step of the pipeline the pages
// describe (thorstenmeyerai.com, pipeline steps "Infer once" / "Select top-K";
// aimodeling.com "First cut": top-100 probabilities cached for every token),
// here over logits that are already on the device.
//
// One block of 512 threads per row (grid-stride over rows, several blocks per
// SM); the row is read from HBM once (16-byte loads, several in flight per
// thread) and a second time from L2:
//   pass 1  per-slot maximum key (1024 slots: two per thread, every element in
//           exactly one) and an online (max, sum of 2^x) for lse;
//   select  theta = the K-th largest slot maximum, by a binary search over the
//           key space with block-wide counts: at least K distinct elements
//           reach theta, so every top-K element has key >= theta;
//   pass 2  collect the elements with key >= theta (typically a few hundred)
//           into shared memory; rank them by (key descending, id ascending)
//           by counting (bitonic sort above 1024 candidates);
//   fallback  when more than CACHE_CAP elements reach theta (heavily tied or
//           adversarial rows) the exact K-th key is found by a binary search
//           over the key space, and the tied elements at it are taken in
//           ascending id order by an ordered block scan.
// Keys are the order-preserving unsigned images of the logits (sign bit
// flipped for positives, all bits for negatives, -0 folded onto +0), so
// comparisons are exact and equal logits have equal keys.
#pragma once

#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include <type_traits>

#include "kd_ptx.cuh"
#include "kdtopk.h"

namespace kd {

constexpr int CACHE_THREADS = 512;
constexpr int CACHE_SLOTS = 2 * CACHE_THREADS;  // per-row maxima used to bound the K-th key
constexpr int CACHE_CAP = 4096;                 // candidates kept in shared memory
constexpr int CACHE_UNROLL = 4;                 // 16-byte loads in flight per thread

template <typename T>
struct LogitTraits;

// key(x): the order-preserving unsigned image of a logit; fkey(f) the same for
// a float holding a value of the type; kvalue(k) the value whose key is k.
template <>
struct LogitTraits<float> {
  static constexpr int KEY_BITS = 32;
  static constexpr int PER_VEC = 4;  // elements per 16-byte load
  __device__ static float value(float x) { return x; }
  __device__ static uint32_t fkey(float x) {
    uint32_t b = __float_as_uint(x);
    if (b == 0x80000000u) b = 0u;  // -0 == +0
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  }
  __device__ static uint32_t key(float x) { return fkey(x); }
  __device__ static float kvalue(uint32_t k) { return __uint_as_float((k & 0x80000000u) ? (k ^ 0x80000000u) : ~k); }
  // the 4 floats of a 16-byte group
  __device__ static void unpack(const uint4& r, float (&f)[4]) {
    f[0] = __uint_as_float(r.x);
    f[1] = __uint_as_float(r.y);
    f[2] = __uint_as_float(r.z);
    f[3] = __uint_as_float(r.w);
  }
  // maximum of a 16-byte group (screening only: -0 and +0 compare equal)
  __device__ static float group_max(const uint4& r) {
    return fmaxf(fmaxf(__uint_as_float(r.x), __uint_as_float(r.y)), fmaxf(__uint_as_float(r.z), __uint_as_float(r.w)));
  }
};

template <>
struct LogitTraits<__nv_bfloat16> {
  static constexpr int KEY_BITS = 16;
  static constexpr int PER_VEC = 8;
  __device__ static float value(__nv_bfloat16 x) { return __bfloat162float(x); }
  __device__ static uint32_t fkey(float x) {  // x holds a bf16 value exactly
    uint32_t b = __float_as_uint(x) >> 16;
    if (b == 0x8000u) b = 0u;  // -0 == +0
    return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
  }
  __device__ static uint32_t key(__nv_bfloat16 x) { return fkey(__bfloat162float(x)); }
  __device__ static float kvalue(uint32_t k) {
    const uint32_t b = (k & 0x8000u) ? (k ^ 0x8000u) : (~k & 0xFFFFu);
    return __uint_as_float(b << 16);
  }
  // the 8 bf16 values of a 16-byte group as floats (bf16 = the top half of an fp32)
  __device__ static void unpack(const uint4& r, float (&f)[8]) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      f[2 * i] = __uint_as_float(w[i] << 16);
      f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  // maximum of a 16-byte group by packed bf16 max (screening only)
  __device__ static float group_max(const uint4& r) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&r);
    const __nv_bfloat162 a = __hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3]));
    return fmaxf(__low2float(a), __high2float(a));
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

// Online softmax normaliser over logits x (natural units): (m, s) with
// m the running maximum and s = sum 2^((x - m) log2 e); -inf logits add nothing.
template <int N>
__device__ __forceinline__ void lse_fold(float& m, float& s, float xmax, const float (&x)[N]) {
  if (xmax == -INFINITY) return;
  if (xmax > m) {
    s *= ex2((m - xmax) * kLog2e);
    m = xmax;
  }
  const float nm = -m * kLog2e;
#pragma unroll
  for (int i = 0; i < N; ++i) s += ex2(fmaf(x[i], kLog2e, nm));
}

__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  const float mn = fmaxf(m, m2);
  s = (mn == -INFINITY) ? 0.f : s * ex2((m - mn) * kLog2e) + s2 * ex2((m2 - mn) * kLog2e);
  m = mn;
}

// Element-wise access to one row, as 16-byte vectors when the row allows it;
// a loaded group stays packed (Raw) until its elements are used.
template <typename TL, bool VEC>
struct RowView {
  const TL* z;
  int V;
  static constexpr int PV = VEC ? LogitTraits<TL>::PER_VEC : 1;
  using Raw = typename std::conditional<VEC, uint4, TL>::type;
  __device__ int groups() const { return VEC ? V / PV : V; }
  __device__ Raw load(int g) const {
    if constexpr (VEC) return __ldg(reinterpret_cast<const uint4*>(z) + g);
    else return z[g];
  }
  __device__ static TL elem(const Raw& r, int i) {
    if constexpr (VEC) return reinterpret_cast<const TL*>(&r)[i];
    else return r;
  }
  __device__ static void floats(const Raw& r, float (&f)[PV]) {
    if constexpr (VEC) LogitTraits<TL>::unpack(r, f);
    else f[0] = LogitTraits<TL>::value(r);
  }
};

template <typename TL, bool VEC>
__global__ void __launch_bounds__(CACHE_THREADS, 2)
    kd_topk_cache_kernel(const TL* __restrict__ Z, int64_t T, int V, int K, int32_t* __restrict__ idx_out,
                         float* __restrict__ p_out, float* __restrict__ lse_out) {
  using Tr = LogitTraits<TL>;
  using RV = RowView<TL, VEC>;
  constexpr int PV = RV::PV;
  __shared__ uint64_t cand[CACHE_CAP];  // (~key << 32) | id: ascending = key descending, id ascending
  __shared__ float red_m[32], red_s[32];
  __shared__ int red_i[32];
  __shared__ int s_count;
  __shared__ float s_lse;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  constexpr int NW = CACHE_THREADS / 32;

  for (int64_t row = blockIdx.x; row < T; row += gridDim.x) {
    const RV rv{Z + row * static_cast<int64_t>(V), V};
    const int ng = rv.groups();
    // ---------------- pass 1: slot maxima, online softmax normaliser
    float fslot0 = -INFINITY, fslot1 = -INFINITY;  // two disjoint element sets per thread
    float m = -INFINITY, s = 0.f;
    int it = 0;
    for (int g0 = tid; g0 < ng; g0 += CACHE_THREADS * CACHE_UNROLL, ++it) {
      if (g0 + (CACHE_UNROLL - 1) * CACHE_THREADS < ng) {
        // all groups present: one rescale check for CACHE_UNROLL * PV logits
        typename RV::Raw x[CACHE_UNROLL];
#pragma unroll
        for (int u = 0; u < CACHE_UNROLL; ++u) x[u] = rv.load(g0 + u * CACHE_THREADS);
        float f[CACHE_UNROLL * PV];
#pragma unroll
        for (int u = 0; u < CACHE_UNROLL; ++u) {
          float fu[PV];
          RV::floats(x[u], fu);
#pragma unroll
          for (int i = 0; i < PV; ++i) f[u * PV + i] = fu[i];
        }
        float fmx = f[0];
#pragma unroll
        for (int i = 1; i < CACHE_UNROLL * PV; ++i) fmx = fmaxf(fmx, f[i]);
        lse_fold(m, s, fmx, f);
        if (it & 1) fslot1 = fmaxf(fslot1, fmx);
        else fslot0 = fmaxf(fslot0, fmx);
      } else {
        for (int u = 0; u < CACHE_UNROLL && g0 + u * CACHE_THREADS < ng; ++u) {
          float f[PV];
          RV::floats(rv.load(g0 + u * CACHE_THREADS), f);
          float fmx = f[0];
#pragma unroll
          for (int i = 1; i < PV; ++i) fmx = fmaxf(fmx, f[i]);
          lse_fold(m, s, fmx, f);
          if (it & 1) fslot1 = fmaxf(fslot1, fmx);
          else fslot0 = fmaxf(fslot0, fmx);
        }
      }
    }
    if constexpr (VEC) {  // the tail that does not fill a 16-byte vector
      for (int j = ng * PV + tid; j < V; j += CACHE_THREADS) {
        const float f[1] = {Tr::value(rv.z[j])};
        lse_fold(m, s, f[0], f);
        fslot1 = fmaxf(fslot1, f[0]);
      }
    }
    // slots without elements hold -inf: no larger than any element, so they never raise theta
    const uint32_t kslot0 = Tr::fkey(fslot0), kslot1 = Tr::fkey(fslot1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lse_merge(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
    __syncthreads();  // the previous row's shared state is no longer read
    if (lane == 0) {
      red_m[warp] = m;
      red_s[warp] = s;
    }
    if (tid == 0) s_count = 0;
    __syncthreads();
    if (warp == 0) {
      float mm = lane < NW ? red_m[lane] : -INFINITY;
      float ss = lane < NW ? red_s[lane] : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) lse_merge(mm, ss, __shfl_xor_sync(0xffffffffu, mm, o), __shfl_xor_sync(0xffffffffu, ss, o));
      if (lane == 0) s_lse = mm + log2f(ss) * kLn2;
    }
    // ---------------- theta: the K-th largest of the 1024 slot maxima (slots
    // without elements hold key 0, the smallest key)
    uint64_t lo = 0, hi = (Tr::KEY_BITS == 32) ? 0xFFFFFFFFull : 0xFFFFull;
    while (lo < hi) {
      const uint64_t mid = lo + (hi - lo + 1) / 2;
      const int c = __syncthreads_count(kslot0 >= mid) + __syncthreads_count(kslot1 >= mid);
      if (c >= K) lo = mid;
      else hi = mid - 1;
    }
    const uint32_t theta = static_cast<uint32_t>(lo);

    // ---------------- pass 2: candidates with key >= theta, i.e. value >= theta's value
    const float tv = Tr::kvalue(theta);
    for (int g0 = tid; g0 < ng; g0 += CACHE_THREADS * CACHE_UNROLL) {
      typename RV::Raw x[CACHE_UNROLL];
#pragma unroll
      for (int u = 0; u < CACHE_UNROLL; ++u)
        if (g0 + u * CACHE_THREADS < ng) x[u] = rv.load(g0 + u * CACHE_THREADS);
#pragma unroll
      for (int u = 0; u < CACHE_UNROLL; ++u) {
        const int g = g0 + u * CACHE_THREADS;
        if (g >= ng) break;
        if constexpr (VEC) {
          if (!(Tr::group_max(x[u]) >= tv)) continue;  // the common case: no candidate in the group
        }
        float f[PV];
        RV::floats(x[u], f);
#pragma unroll
        for (int i = 0; i < PV; ++i) {
          if (f[i] >= tv) {
            const int at = atomicAdd(&s_count, 1);
            if (at < CACHE_CAP)
              cand[at] = (static_cast<uint64_t>(~Tr::fkey(f[i])) << 32) | static_cast<uint32_t>(g * PV + i);
          }
        }
      }
    }
    if constexpr (VEC) {
      for (int j = ng * PV + tid; j < V; j += CACHE_THREADS) {
        const float f = Tr::value(rv.z[j]);
        if (f >= tv) {
          const int at = atomicAdd(&s_count, 1);
          if (at < CACHE_CAP) cand[at] = (static_cast<uint64_t>(~Tr::fkey(f)) << 32) | static_cast<uint32_t>(j);
        }
      }
    }
    __syncthreads();
    int n = s_count;
    if (n > CACHE_CAP) {
      // ---------------- fallback: exact K-th key by binary search, then ordered ties
      // largest kappa with count(key >= kappa) >= K, searched in [theta, 2^bits - 1]
      uint64_t lo2 = theta, hi2 = (Tr::KEY_BITS == 32) ? 0xFFFFFFFFull : 0xFFFFull;
      while (lo2 < hi2) {
        const uint64_t mid = lo2 + (hi2 - lo2 + 1) / 2;
        int c = 0;
        for (int j = tid; j < V; j += CACHE_THREADS) c += static_cast<uint64_t>(Tr::key(rv.z[j])) >= mid;
        if (block_sum_int(c, red_i) >= K) lo2 = mid;
        else hi2 = mid - 1;
      }
      const uint32_t kappa = static_cast<uint32_t>(lo2);
      __syncthreads();
      if (tid == 0) s_count = 0;
      __syncthreads();
      for (int j = tid; j < V; j += CACHE_THREADS) {  // fewer than K are strictly above kappa
        const uint32_t k = Tr::key(rv.z[j]);
        if (k > kappa) cand[atomicAdd(&s_count, 1)] = (static_cast<uint64_t>(~k) << 32) | static_cast<uint32_t>(j);
      }
      __syncthreads();
      int taken = s_count;
      // ties at kappa in ascending id order, one block-wide segment at a time
      for (int base = 0; base < V && taken < K; base += CACHE_THREADS) {
        const int j = base + tid;
        const bool tie = j < V && Tr::key(rv.z[j]) == kappa;
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
    // ---------------- order the candidates and emit the top K
    const float lse = s_lse;
    if (n <= 2 * CACHE_THREADS) {
      // rank of each candidate = number of smaller composite keys (all distinct)
      uint64_t mine[2];
      int rank[2] = {0, 0};
#pragma unroll
      for (int h = 0; h < 2; ++h) mine[h] = (tid + h * CACHE_THREADS < n) ? cand[tid + h * CACHE_THREADS] : ~0ull;
      if (tid < n) {  // only candidate owners count
        if (tid + CACHE_THREADS < n) {
          for (int j = 0; j < n; ++j) {
            const uint64_t c = cand[j];
            rank[0] += c < mine[0];
            rank[1] += c < mine[1];
          }
        } else {
          for (int j = 0; j < n; ++j) rank[0] += cand[j] < mine[0];
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (tid + h * CACHE_THREADS < n && rank[h] < K) {
          const int id = static_cast<int>(mine[h] & 0xFFFFFFFFu);
          idx_out[row * K + rank[h]] = id;
          p_out[row * K + rank[h]] = ex2((Tr::value(rv.z[id]) - lse) * kLog2e);
        }
      }
    } else {
      int n_pad = 1;
      while (n_pad < n) n_pad <<= 1;
      for (int i = n + tid; i < n_pad; i += CACHE_THREADS) cand[i] = ~0ull;
      __syncthreads();
      block_bitonic_sort_u64(cand, n_pad);
      for (int k = tid; k < K; k += CACHE_THREADS) {
        const int id = static_cast<int>(cand[k] & 0xFFFFFFFFu);
        idx_out[row * K + k] = id;
        p_out[row * K + k] = ex2((Tr::value(rv.z[id]) - lse) * kLog2e);
      }
    }
    if (tid == 0 && lse_out) lse_out[row] = lse;
  }
}

}  // namespace kd
