// Offline teacher-cache builder: for each row of teacher logits Z[T, V] the K
// largest logits' ids (largest first, equal logits by ascending id) and their
// softmax probabilities p = exp(z - lse) (so the row's mass M_t = sum_k p <= 1).
// This is the "keep the top-100 of every token" step of the pipeline the pages
// describe (thorstenmeyerai.com, pipeline steps "Infer once" / "Select top-K";
// aimodeling.com "First cut": top-100 probabilities cached for every token),
// here over logits that are already on the device.
//
// One block per row (grid-stride over rows): 256-thread blocks, four per SM,
// for rows of up to 512 KB (256 KB when they are read 16 bytes at a time),
// 512-thread blocks, two per SM, for longer rows (the block shapes below).
// Each row is read from HBM once, with 32-byte loads (one 256-bit load) when
// the row is a whole number of 32-byte groups on a 32-byte boundary, 16-byte
// loads otherwise, several in flight per thread, behind L2 prefetches that
// keep a window of the row requested ahead of pass 1 (48 KB for the narrow
// shape with 32-byte loads, 64 KB with 16-byte loads, 128 KB for the wide one; the wide shape requests a row of up to
// 256 KB whole).  The head of the block's next row is requested while the
// block selects this one, so that HBM keeps streaming through the selection:
//   pass 1  per-slot maximum (two slots per thread, every element in
//           exactly one), an online (max, sum of 2^x) for lse, and the maximum
//           of every load's group (32 or 16 bytes), kept in shared memory (as
//           bf16, rounded up for fp32 logits);
//   select  theta = the K-th largest slot maximum, by a byte-wise radix select
//           over 256-bin shared-memory histograms (with the block's lse
//           reduced alongside): at least K distinct elements reach theta, so
//           every top-K element has key >= theta;
//   pass 2  only the groups whose maximum reaches theta (typically about K of
//           them) are listed and read again (from L2, unless the narrow
//           shape's window has moved on), all in flight together,
//           and their elements >= theta are collected in shared memory (list
//           and candidates appended with one atomic per warp); they are
//           ranked by (key descending, id ascending) by counting (bitonic
//           sort above two candidates per thread);
//   fallback  rows whose group maxima do not fit in shared memory, or that
//           cannot be read 16 bytes at a time, are scanned whole in pass 2;
//           when more candidates reach theta than the list holds (heavily tied or
//           adversarial rows) the exact K-th key is found by a binary search
//           over the key space, and the tied elements at it are taken in
//           ascending id order by an ordered block scan.
// Keys are the order-preserving unsigned images of the logits (sign bit
// flipped for positives, all bits for negatives, -0 folded onto +0), so
// comparisons are exact and equal logits have equal keys.  A candidate is the
// composite (~key << 32 | id): ascending composites are the output order, and
// the logit is recovered from the key, so p needs no second read of Z.
#pragma once

#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include <type_traits>

#include "kd_ptx.cuh"
#include "kdtopk.h"

namespace kd {

constexpr int CACHE_UNROLL = 4;              // loads in flight per thread, rows read element-wise
constexpr int CACHE_GLIST = 1024;            // groups listed for the re-read of pass 2
constexpr int64_t CACHE_WHOLE_ROW = 262144;  // the wide shape prefetches rows up to this many bytes whole

// Block shapes.  The narrow shape (256-thread blocks, four per SM, each row
// requested into L2 through a 48 or 64 KB window, since four resident rows per SM
// requested whole would not fit in L2) takes rows whose group maxima fit its
// shared memory: up to 512 KB read 32 bytes at a time, 256 KB read 16 bytes at
// a time, when K is at most its slot count.  The wide shape (512-thread
// blocks, two per SM, a row of up to 256 KB requested whole, a longer one
// through a 128 KB window) takes the rest.  CAP candidates and GMAX group
// maxima are kept in shared memory; HEAD bytes of the block's next row are
// requested while it selects a row.
template <int NT_, int MINB_, int CAP_, int GMAX_, bool ALL_WINDOWED_, int64_t WINDOW_, int64_t HEAD_, int VB_ = 16>
struct CacheShape {
  static constexpr int NT = NT_;
  static constexpr int MINB = MINB_;
  static constexpr int CAP = CAP_;
  static constexpr int GMAX = GMAX_;
  static constexpr bool ALL_WINDOWED = ALL_WINDOWED_;
  static constexpr int64_t WINDOW = WINDOW_;
  static constexpr int64_t HEAD = HEAD_;
  static constexpr int SLOTS = 2 * NT_;  // slot maxima per row: theta needs K <= SLOTS
  // bytes per vector load of rows read in vectors (16, or 32 with one group
  // maximum per 32 bytes), and vector loads in flight per thread
  static constexpr int VB = VB_;
  static constexpr int UNR = VB_ == 32 ? 2 : 4;
  // dynamic shared memory: the candidate list, and the group maxima when rows
  // are read 16 bytes at a time
  static constexpr int smem_bytes(bool vec) { return CAP * 8 + (vec ? GMAX * 2 : 0); }
};
using CacheNarrow = CacheShape<256, 4, 2048, 16384, true, 65536, 32768>;
using CacheNarrow32 = CacheShape<256, 4, 2048, 16384, true, 49152, 16384, 32>;
using CacheWide = CacheShape<512, 2, 4096, 32768, false, 131072, 65536>;
using CacheWide32 = CacheShape<512, 2, 4096, 32768, false, 131072, 65536, 32>;

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
  // maximum of a 32-byte group
  __device__ static float group_max2(const uint4& a, const uint4& b) { return fmaxf(group_max(a), group_max(b)); }
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
  // maximum of a 32-byte group
  __device__ static float group_max2(const uint4& a, const uint4& b) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* k = reinterpret_cast<const __nv_bfloat162*>(&b);
    const __nv_bfloat162 x = __hmax2(__hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3])),
                                     __hmax2(__hmax2(k[0], k[1]), __hmax2(k[2], k[3])));
    return fmaxf(__low2float(x), __high2float(x));
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

// Merges two online softmax normalisers (m, s) over logits in natural units:
// s = sum 2^((x - m) log2 e) over the logits seen, m their running maximum.
__device__ __forceinline__ void lse_merge(float& m, float& s, float m2, float s2) {
  const float mn = fmaxf(m, m2);
  s = (mn == -INFINITY) ? 0.f : s * ex2((m - mn) * kLog2e) + s2 * ex2((m2 - mn) * kLog2e);
  m = mn;
}

// 32 bytes of a row, loaded by one 256-bit load
struct Vec32 {
  uint4 a, b;
};

__device__ __forceinline__ Vec32 ldg_v32(const void* p) {
  Vec32 r;
  asm("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(r.a.x), "=r"(r.a.y), "=r"(r.a.z), "=r"(r.a.w), "=r"(r.b.x), "=r"(r.b.y), "=r"(r.b.z), "=r"(r.b.w)
      : "l"(p));
  return r;
}

// Element-wise access to one row, as VB-byte vectors (16 or 32) when the row
// allows it; a loaded group stays packed (Raw) until its elements are used.
template <typename TL, bool VEC, int VB = 16>
struct RowView {
  const TL* z;
  int V;
  static constexpr int PV16 = LogitTraits<TL>::PER_VEC;  // elements per 16 bytes
  static constexpr int PV = VEC ? PV16 * (VB / 16) : 1;
  using Raw = typename std::conditional<VEC, typename std::conditional<VB == 32, Vec32, uint4>::type, TL>::type;
  __device__ int groups() const { return VEC ? V / PV : V; }  // VEC rows are whole groups
  __device__ Raw load(int g) const {
    if constexpr (VEC && VB == 32) return ldg_v32(reinterpret_cast<const char*>(z) + static_cast<size_t>(g) * 32);
    else if constexpr (VEC) return __ldg(reinterpret_cast<const uint4*>(z) + g);
    else return z[g];
  }
  __device__ static TL elem(const Raw& r, int i) {
    if constexpr (VEC) return reinterpret_cast<const TL*>(&r)[i];
    else return r;
  }
  __device__ static void floats(const Raw& r, float (&f)[PV]) {
    if constexpr (VEC && VB == 32) {
      LogitTraits<TL>::unpack(r.a, *reinterpret_cast<float(*)[PV16]>(&f[0]));
      LogitTraits<TL>::unpack(r.b, *reinterpret_cast<float(*)[PV16]>(&f[PV16]));
    } else if constexpr (VEC) {
      LogitTraits<TL>::unpack(r, f);
    } else {
      f[0] = LogitTraits<TL>::value(r);
    }
  }
  // the largest value of a loaded group
  __device__ static float gmax(const Raw& r) {
    if constexpr (VEC && VB == 32) return LogitTraits<TL>::group_max2(r.a, r.b);
    else if constexpr (VEC) return LogitTraits<TL>::group_max(r);
    else return LogitTraits<TL>::value(r);
  }
};

// Appends the candidate (key, id) to the block's list; entries past CAP are
// counted but not stored.
template <int CAP>
__device__ __forceinline__ void push_cand(uint64_t* cand, int* count, uint32_t key, int id) {
  const int at = atomicAdd(count, 1);
  if (at < CAP) cand[at] = (static_cast<uint64_t>(~key) << 32) | static_cast<uint32_t>(id);
}

// Reserves n >= 0 consecutive slots of a shared counter for each lane of the
// warp (all 32 lanes call it) with one atomic per warp; returns the lane's
// first slot.
__device__ __forceinline__ int warp_reserve(int* counter, int n) {
  const int lane = threadIdx.x & 31;
  int incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  const int total = __shfl_sync(0xffffffffu, incl, 31);
  int base = 0;
  if (lane == 31 && total) base = atomicAdd(counter, total);
  return __shfl_sync(0xffffffffu, base, 31) + incl - n;
}

// One byte-level step of a most-significant-byte-first radix select of the
// K-th largest of the block's keys (two per thread), after
// every thread has counted its keys that share `prefix` into hist[256] by the
// byte at `shift` and the block has synchronised.  Warp 0 picks the byte b of
// the K-th largest, stores (b, keys above b's bin) in sel[0..1] and clears
// hist for its next use; the caller synchronises before reading sel.
__device__ __forceinline__ void radix_pick(int* hist, int* sel, int need) {
  const int lane = threadIdx.x & 31;
  int h[8];
  int sum = 0;
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    h[b] = hist[lane * 8 + b];
    hist[lane * 8 + b] = 0;
    sum += h[b];
  }
  int incl = sum;  // keys in the bins of lanes >= lane
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_down_sync(0xffffffffu, incl, o);
    if (lane + o < 32) incl += v;
  }
  const int above = incl - sum;  // keys in the bins of lanes > lane
  if (above < need && incl >= need) {
    int acc = above;
#pragma unroll
    for (int b = 7; b >= 0; --b) {
      if (acc + h[b] >= need) {
        sel[0] = lane * 8 + b;
        sel[1] = acc;
        break;
      }
      acc += h[b];
    }
  }
}

// Counts key k into hist by its byte at `shift` when its bytes above `shift`
// equal `prefix`.
template <int KEY_BITS>
__device__ __forceinline__ void radix_count(uint32_t k, int shift, uint32_t prefix, int* hist) {
  const int hs = shift + 8;
  if (hs >= KEY_BITS || (k >> hs) == prefix) atomicAdd(&hist[(k >> shift) & 255], 1);
}

// bf16 bits of a group maximum, never below it: exact for bf16 logits,
// rounded up for fp32 ones (a group is re-read when this reaches theta).
template <typename TL>
__device__ __forceinline__ uint16_t gmax_bits(float x) {
  if constexpr (std::is_same<TL, __nv_bfloat16>::value) return static_cast<uint16_t>(__float_as_uint(x) >> 16);
  else return __bfloat16_as_ushort(__float2bfloat16_ru(x));
}

// Statistics of U loaded groups x[0..U): the slot maxima (load u feeds slot
// u % 2), the online normaliser (m, s), folded group after group, and each
// group's maximum in gm[u].
template <int U, typename RV>
__device__ __forceinline__ void groups_stats(const typename RV::Raw (&x)[U], float (&gm)[U], float& m, float& s,
                                             float& slot0, float& slot1) {
  constexpr int PV = RV::PV;
  float fmx = -INFINITY;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    gm[u] = RV::gmax(x[u]);
    fmx = fmaxf(fmx, gm[u]);
    if (u & 1) slot1 = fmaxf(slot1, gm[u]);  // load u of an iteration feeds slot u % 2
    else slot0 = fmaxf(slot0, gm[u]);
  }
  if (fmx == -INFINITY) return;  // -inf logits add nothing
  if (fmx > m) {
    s *= ex2((m - fmx) * kLog2e);
    m = fmx;
  }
  const float nm = -m * kLog2e;
  if constexpr (PV == 1) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float f[1];
      RV::floats(x[u], f);
      s += ex2(fmaf(f[0], kLog2e, nm));
    }
  } else {
    // two logits per packed fp32 FMA / add (Blackwell f32x2)
    const float2 l2 = make_float2(kLog2e, kLog2e), nm2 = make_float2(nm, nm);
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float f[PV];
      RV::floats(x[u], f);
#pragma unroll
      for (int i = 0; i < PV; i += 2) {
        const float2 t = __ffma2_rn(make_float2(f[i], f[i + 1]), l2, nm2);
        acc = __fadd2_rn(acc, make_float2(ex2(t.x), ex2(t.y)));
      }
    }
    s += acc.x + acc.y;
  }
}

template <typename TL, bool VEC, typename S>
__global__ void __launch_bounds__(S::NT, S::MINB)
    kd_topk_cache_kernel(const TL* __restrict__ Z, int64_t T, int V, int K, int32_t* __restrict__ idx_out,
                         float* __restrict__ p_out, float* __restrict__ lse_out) {
  using Tr = LogitTraits<TL>;
  using RV = RowView<TL, VEC, S::VB>;
  constexpr int UNR = VEC ? S::UNR : CACHE_UNROLL;  // loads in flight per thread
  constexpr int PV = RV::PV;
  constexpr int NW = S::NT / 32;
  extern __shared__ __align__(16) unsigned char cache_smem[];
  uint64_t* cand = reinterpret_cast<uint64_t*>(cache_smem);  // (~key << 32) | id
  uint16_t* gmax = reinterpret_cast<uint16_t*>(cache_smem + S::CAP * 8);  // used when VEC
  __shared__ float red_m[32], red_s[32];
  __shared__ int red_i[32];
  __shared__ int hist[256];  // radix-select counts, zero between uses
  __shared__ int sel[2];
  __shared__ int glist[CACHE_GLIST];  // groups re-read in pass 2
  __shared__ int s_count, s_groups;
  __shared__ float s_lse;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < 256; i += S::NT) hist[i] = 0;

  const int64_t row_bytes = static_cast<int64_t>(V) * sizeof(TL);
  const bool windowed = VEC && (S::ALL_WINDOWED || row_bytes > CACHE_WHOLE_ROW);
  // thread 0: bytes of the current row already requested into L2, and of the
  // block's next row (its head, requested during this row's selection)
  int64_t req = 0, req_next = 0;
  auto request_upto = [&](const TL* rz, int64_t upto) {  // multiples of 16 bytes, within the row
    upto = min(upto, row_bytes);
    if (upto > req) {
      prefetch_l2_bulk(reinterpret_cast<const char*>(rz) + req, upto - req);
      req = upto;
    }
  };
  for (int64_t row = blockIdx.x; row < T; row += gridDim.x) {
    const RV rv{Z + row * static_cast<int64_t>(V), V};
    const int ng = rv.groups();
    const bool screen = VEC && ng <= S::GMAX;  // group maxima fit in shared memory
    if constexpr (VEC) {
      if (tid == 0) {
        req = req_next;
        req_next = 0;
        request_upto(rv.z, windowed ? S::WINDOW : row_bytes);
      }
    }
    // ---------------- pass 1: slot maxima, online softmax normaliser, group maxima
    float fslot0 = -INFINITY, fslot1 = -INFINITY;  // two disjoint element sets per thread
    float m = -INFINITY, s = 0.f;
    int it = 0;
    for (int g0 = tid; g0 < ng; g0 += S::NT * UNR, ++it) {
      // keep the window ahead of what this iteration reads (VB bytes per group)
      if (windowed && tid == 0)
        request_upto(rv.z, static_cast<int64_t>(it + 1) * S::NT * UNR * S::VB + S::WINDOW);
      if (g0 + (UNR - 1) * S::NT < ng) {
        typename RV::Raw x[UNR];
        float gm[UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u) x[u] = rv.load(g0 + u * S::NT);
        groups_stats<UNR, RV>(x, gm, m, s, fslot0, fslot1);
        if (screen) {
#pragma unroll
          for (int u = 0; u < UNR; ++u) gmax[g0 + u * S::NT] = gmax_bits<TL>(gm[u]);
        }
      } else {
        for (int u = 0; u < UNR && g0 + u * S::NT < ng; ++u) {
          const typename RV::Raw x[1] = {rv.load(g0 + u * S::NT)};
          float gm[1];
          groups_stats<1, RV>(x, gm, m, s, fslot0, fslot1);
          if (screen) gmax[g0 + u * S::NT] = gmax_bits<TL>(gm[0]);
        }
      }
    }
    // (rows read in vectors are whole groups: there is no tail)
    // slots without elements hold -inf: no larger than any element, so they never raise theta
    const uint32_t kslot0 = Tr::fkey(fslot0), kslot1 = Tr::fkey(fslot1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lse_merge(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
    __syncthreads();  // the previous row's shared state is no longer read (and hist is clear)
    // ---------------- theta: the K-th largest of the slot maxima, by radix
    // select one byte at a time; the block's lse is reduced alongside
    if (lane == 0) {
      red_m[warp] = m;
      red_s[warp] = s;
    }
    if (tid == 0) {
      s_count = 0;
      s_groups = 0;
    }
    uint32_t prefix = 0;  // the bytes of theta found so far
    int need = K;         // theta's rank among the keys that share them
#pragma unroll
    for (int shift = Tr::KEY_BITS - 8; shift >= 0; shift -= 8) {
      radix_count<Tr::KEY_BITS>(kslot0, shift, prefix, hist);
      radix_count<Tr::KEY_BITS>(kslot1, shift, prefix, hist);
      __syncthreads();
      if (warp == 0) {
        radix_pick(hist, sel, need);
        if (shift == Tr::KEY_BITS - 8) {
          float mm = lane < NW ? red_m[lane] : -INFINITY;
          float ss = lane < NW ? red_s[lane] : 0.f;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1)
            lse_merge(mm, ss, __shfl_xor_sync(0xffffffffu, mm, o), __shfl_xor_sync(0xffffffffu, ss, o));
          if (lane == 0) s_lse = mm + log2f(ss) * kLn2;
        }
      }
      __syncthreads();
      prefix = (prefix << 8) | static_cast<uint32_t>(sel[0]);
      need -= sel[1];
    }
    const uint32_t theta = prefix;
    if constexpr (VEC) {
      // the head of the block's next row into L2 while this row's selection runs
      if (tid == 0 && row + gridDim.x < T) {
        req_next = min(row_bytes, S::HEAD);
        prefetch_l2_bulk(rv.z + static_cast<int64_t>(gridDim.x) * V, req_next);
      }
    }

    // ---------------- pass 2: every element with key >= theta, i.e. value >= theta's value
    const float tv = Tr::kvalue(theta);
    if (screen) {
      // only the groups whose maximum reaches theta, listed first so that their
      // re-reads (from L2) are all in flight together
      // eight maxima per 16-byte read, compared as packed bf16 against the
      // smallest bf16 >= theta's value
      const __nv_bfloat162 th2 = __bfloat162bfloat162(__float2bfloat16_ru(tv));
      const int nv = (ng + 7) / 8;
      for (int v = tid; v < nv; v += S::NT) {
        const uint4 w = reinterpret_cast<const uint4*>(gmax)[v];
        // the common case first: none of the eight maxima reaches theta (entries
        // past the row's end may hold anything; the exact mask below drops them)
        const __nv_bfloat162* h8 = reinterpret_cast<const __nv_bfloat162*>(&w);
        if (!__hge2_mask(__hmax2(__hmax2(h8[0], h8[1]), __hmax2(h8[2], h8[3])), th2)) continue;
        const uint32_t h0 = __hge2_mask(h8[0], th2), h1 = __hge2_mask(h8[1], th2);
        const uint32_t h2 = __hge2_mask(h8[2], th2), h3 = __hge2_mask(h8[3], th2);
        uint32_t m8 = (h0 & 1u) | ((h0 >> 15) & 2u) | ((h1 & 1u) << 2) | ((h1 >> 13) & 8u) | ((h2 & 1u) << 4) |
                      ((h2 >> 11) & 32u) | ((h3 & 1u) << 6) | ((h3 >> 9) & 128u);  // bit e: group v * 8 + e
        if (v * 8 + 8 > ng) m8 &= (1u << (ng - v * 8)) - 1u;  // groups past the row's end
        if (!m8) continue;
        int at = atomicAdd(&s_groups, __popc(m8));  // one shared atomic per lane with hits
        for (; m8; m8 &= m8 - 1u, ++at) {
          const int g = v * 8 + __ffs(m8) - 1;
          if (at < CACHE_GLIST) {
            glist[at] = g;
          } else {  // a long list: this group now
            float f[PV];
            RV::floats(rv.load(g), f);
#pragma unroll
            for (int e = 0; e < PV; ++e)
              if (f[e] >= tv) push_cand<S::CAP>(cand, &s_count, Tr::fkey(f[e]), g * PV + e);
          }
        }
      }
      __syncthreads();
      const int nl = min(s_groups, CACHE_GLIST);
      for (int i0 = warp * 32; i0 < nl; i0 += S::NT) {  // i = tid + k S::NT
        const int i = i0 + lane;
        const int g = i < nl ? glist[i] : 0;
        float f[PV];
        uint32_t mk = 0;  // bit e: element e of the group reaches theta
        if (i < nl) {
          RV::floats(rv.load(g), f);
#pragma unroll
          for (int e = 0; e < PV; ++e) mk |= static_cast<uint32_t>(f[e] >= tv) << e;
        }
        int at = warp_reserve(&s_count, __popc(mk));
#pragma unroll
        for (int e = 0; e < PV; ++e)
          if ((mk >> e) & 1u) {
            if (at < S::CAP) cand[at] = (static_cast<uint64_t>(~Tr::fkey(f[e])) << 32) | static_cast<uint32_t>(g * PV + e);
            ++at;
          }
      }
    } else {
      for (int g0 = tid; g0 < ng; g0 += S::NT * UNR) {
        typename RV::Raw x[UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u)
          if (g0 + u * S::NT < ng) x[u] = rv.load(g0 + u * S::NT);
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
          const int g = g0 + u * S::NT;
          if (g >= ng) break;
          if constexpr (VEC) {
            if (!(RV::gmax(x[u]) >= tv)) continue;  // the common case: no candidate in the group
          }
          float f[PV];
          RV::floats(x[u], f);
#pragma unroll
          for (int i = 0; i < PV; ++i)
            if (f[i] >= tv) push_cand<S::CAP>(cand, &s_count, Tr::fkey(f[i]), g * PV + i);
        }
      }
    }
    __syncthreads();
    int n = s_count;
    if (n > S::CAP) {
      // ---------------- fallback: exact K-th key by binary search, then ordered ties
      // largest kappa with count(key >= kappa) >= K, searched in [theta, 2^bits - 1]
      uint64_t lo2 = theta, hi2 = (Tr::KEY_BITS == 32) ? 0xFFFFFFFFull : 0xFFFFull;
      while (lo2 < hi2) {
        const uint64_t mid = lo2 + (hi2 - lo2 + 1) / 2;
        int cnt = 0;
        for (int j = tid; j < V; j += S::NT) cnt += static_cast<uint64_t>(Tr::key(rv.z[j])) >= mid;
        if (block_sum_int(cnt, red_i) >= K) lo2 = mid;
        else hi2 = mid - 1;
      }
      const uint32_t kappa = static_cast<uint32_t>(lo2);
      __syncthreads();
      if (tid == 0) s_count = 0;
      __syncthreads();
      for (int j = tid; j < V; j += S::NT) {  // fewer than K are strictly above kappa
        const uint32_t k = Tr::key(rv.z[j]);
        if (k > kappa) cand[atomicAdd(&s_count, 1)] = (static_cast<uint64_t>(~k) << 32) | static_cast<uint32_t>(j);
      }
      __syncthreads();
      int taken = s_count;
      // ties at kappa in ascending id order, one block-wide segment at a time
      for (int base = 0; base < V && taken < K; base += S::NT) {
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
    auto emit = [&](uint64_t c, int k) {
      const float z = Tr::kvalue(~static_cast<uint32_t>(c >> 32));
      idx_out[row * K + k] = static_cast<int>(c & 0xFFFFFFFFu);
      p_out[row * K + k] = ex2((z - lse) * kLog2e);
    };
    if (n <= S::NT / 2) {
      // rank of each candidate = number of smaller composite keys (all distinct),
      // counted by P lanes of one warp
      int P = 1;
      while (P < 32 && 2 * P * n <= S::NT) P *= 2;
      const int c = tid / P, part = tid % P;
      const uint64_t mine = c < n ? cand[c] : ~0ull;
      int rank = 0;
      if (c < n) {
#pragma unroll 4
        for (int j = part; j < n; j += P) rank += cand[j] < mine;
      }
      for (int o = 1; o < P; o <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
      if (c < n && part == 0 && rank < K) emit(mine, rank);
    } else if (n <= 2 * S::NT) {
      // rank of each candidate = number of smaller composite keys (all distinct)
      uint64_t mine[2];
      int rank[2] = {0, 0};
#pragma unroll
      for (int h = 0; h < 2; ++h) mine[h] = (tid + h * S::NT < n) ? cand[tid + h * S::NT] : ~0ull;
      if (tid < n) {  // only candidate owners count
        if (tid + S::NT < n) {
          for (int j = 0; j < n; ++j) {
            const uint64_t cj = cand[j];
            rank[0] += cj < mine[0];
            rank[1] += cj < mine[1];
          }
        } else {
          for (int j = 0; j < n; ++j) rank[0] += cand[j] < mine[0];
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h)
        if (tid + h * S::NT < n && rank[h] < K) emit(mine[h], rank[h]);
    } else {
      int n_pad = 1;
      while (n_pad < n) n_pad <<= 1;
      for (int i = n + tid; i < n_pad; i += S::NT) cand[i] = ~0ull;
      __syncthreads();
      block_bitonic_sort_u64(cand, n_pad);
      for (int k = tid; k < K; k += S::NT) emit(cand[k], k);
    }
    if (tid == 0 && lse_out) lse_out[row] = lse;
  }
}

}  // namespace kd
