// Persistent, warp-specialised tcgen05 GEMM for sm_103a:  D[M,N] = A[M,K] B[N,K]^T
// with bf16 operands staged by TMA (128-byte swizzle) into a shared-memory ring
// and fp32 accumulators double-buffered in tensor memory (2 x 256 columns).
//
//   warp 0      TMA producer (one thread)
//   warp 1      tensor-memory allocator and MMA issuer (one thread)
//   warps 2..5  epilogue: thread i of the four warps owns accumulator row i
//
// Two forms, chosen by the PAIR template parameter:
//   single CTA  tile 128 x 256 x 64, 4-stage ring of 48 KB stages;
//   CTA pair    a two-CTA cluster computes a 256 x 256 tile with cta_group::2
//               MMAs issued by the leader CTA: each CTA stages its own 128 rows
//               of A and its own 128 rows of B (32 KB stages, 6-stage ring),
//               the MMA reads B from both CTAs, and each CTA's tensor memory
//               holds its 128 rows of D.  Per MMA flop the pair moves a third
//               less operand data from L2 into shared memory.  The peer's TMA
//               loads signal the leader's "full" barriers; MMA completion is
//               multicast to both CTAs' "empty" / "accumulator full" barriers;
//               the peer's epilogue releases accumulators to the leader.
//
// Tile 128 x 256 x 64 per CTA.  Operands may be K-major (the reduction index is
// contiguous in memory) or MN-major (the row/column index is contiguous); the
// latter lets the backward GEMMs read W, G and H in place.
//
// Epilogues (the loss-specific work happens on the accumulator, in registers):
//   EPI_FWD  logits tile -> per-row online max / sum of exp over the tile's
//            vocabulary columns, plus sum_k p_k z_k over the row's top-K ids
//            that fall inside the tile (sorted ids, one cursor per row).  The
//            logits never leave the SM.
//   EPI_G    logits tile -> G = M_t exp(z - lse_t) - p at the top-K ids,
//            rounded to bf16, staged as 128 x 64 swizzled slices and written
//            by TMA as the [chunk, V] operand of dH / dW (TMA clips the
//            vocabulary tail).
//   EPI_FWD_E  as EPI_FWD, and the tile's exponentials e = 2^(z log2e - m) with
//            m the tile's row maximum are kept: rounded to bf16 and written by
//            TMA into the chunk's [chunk, V] operand buffer, where a later
//            elementwise pass turns them into G once lse is known (the fused
//            step without the backward recompute).
//   EPI_GF   two adjacent chunks in one launch: row tiles below m_split are
//            chunk c's G tiles (EPI_G), the others chunk c+1's forward tiles
//            (EPI_FWD); both halves share every W tile through L2.
//   EPI_F32  fp32 tile, scaled, staged through shared memory (128 x 32 slices,
//            128-byte swizzle) and written by TMA: a plain store, or a TMA
//            reduce-add so that L2 performs the read-modify-write of dW while
//            the next tile's mainloop runs (dW accumulation across chunks,
//            split-K partials of dH, tests).
#pragma once

#include <cuda_bf16.h>
#include <math.h>

#include "kd_ptx.cuh"
#include "kdtopk.h"

namespace kd {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int STAGES = 4;
constexpr int A_STAGE_BYTES = BM * BK * 2;  // 16 KB
constexpr int B_STAGE_BYTES = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
constexpr int TMEM_COLS = 2 * BN;
constexpr int GEMM_THREADS = 192;
constexpr int SMEM_BAR_BYTES = 256;
constexpr int OUT_SLICE_COLS = 32;                        // fp32 columns per TMA output slice
constexpr int OUT_SLICE_BYTES = BM * 128;                 // 16 KB: 128 rows x 128 bytes
constexpr int G_SLICE_COLS = 64;                          // bf16 columns per TMA output slice
constexpr int OUT_STAGING_BYTES = 2 * OUT_SLICE_BYTES;
constexpr int EPI_WARPS = 4;
constexpr uint32_t EPI_BAR_ID = 1;  // named barrier of the epilogue warps

enum Epi { EPI_FWD = 0, EPI_G = 1, EPI_F32 = 2, EPI_FWD_E = 3, EPI_GF = 4 };

__host__ __device__ constexpr int staging_bytes(int epi) { return epi == EPI_FWD ? 0 : OUT_STAGING_BYTES; }

// Per-form shape of the pipeline.
template <bool PAIR>
struct GemmCfg {
  static constexpr int NCTA = PAIR ? 2 : 1;
  static constexpr int TILE_M = BM * NCTA;                  // rows of D per tile
  static constexpr int B_ROWS = BN / NCTA;                  // rows of the B tile one CTA stages
  static constexpr int STAGE = A_STAGE_BYTES + B_ROWS * BK * 2;
  static constexpr int NSTAGE = PAIR ? 6 : STAGES;
};

template <bool PAIR>
__host__ __device__ constexpr size_t gemm_smem_bytes(int epi) {
  return 1024 + size_t(GemmCfg<PAIR>::NSTAGE) * GemmCfg<PAIR>::STAGE + staging_bytes(epi) + SMEM_BAR_BYTES;
}
static_assert(gemm_smem_bytes<true>(EPI_F32) <= 232448, "pair pipeline exceeds the shared-memory limit");
static_assert(gemm_smem_bytes<false>(EPI_F32) <= 232448, "pipeline exceeds the shared-memory limit");

struct GemmParams {
  // tile grid and raster
  int num_m, num_n, num_s;
  int kb_total, kb_per_split;
  int m_fast;  // 1: consecutive tile ids walk m (share a B tile), 0: walk n
  // TMA coordinate offsets, in elements
  int a_mn0, a_k0, b_mn0, b_k0;
  // bounded waits / status
  uint64_t wait_limit_ns;
  int* status;
  int debug_withhold_loads;
  // EPI_FWD / EPI_G
  int rows_valid;
  int V, K;
  const int32_t* sidx;  // [Cpad, K] ids ascending, padded with INT_MAX
  const float* sp;      // [Cpad, K] probabilities in the same order
  float* part_m;        // [num_n, ld_part] base-2 running max (z * log2 e)
  float* part_s;        // [num_n, ld_part] sum of 2^(z log2e - max)
  float* part_pz;       // [num_n, ld_part] sum of p z over ids in the tile
  int ld_part;
  const float* rowM;    // [Cpad] teacher mass per row
  const float* lse;     // [rows_valid] lse of the chunk's rows
  // EPI_F32: output tile (m, n, s) goes to rows out_row0 + s * split_rows + m * BM,
  // columns n * BN of the fp32 tensor map; reduce_add adds instead of storing.
  // EPI_G: tile rows go to out_row0 + m * BM of the G tensor map.
  int out_row0, split_rows;
  int reduce_add;
  float scale;
  // EPI_GF: row tiles m >= m_split are the forward of the next chunk, whose
  // H rows start at a_mn0_2, with rows_valid2 rows and sorted cache sidx2/sp2.
  // EPI_FWD_E with m_split > 0: the forward of two chunks in one launch; the
  // second chunk's kept exponentials go to rows out_row0_2 + ... of the
  // operand buffer and its softmax partials to rows part_row2 + ... of the
  // partial arrays.
  int m_split, a_mn0_2, rows_valid2;
  int out_row0_2, part_row2;
  const int32_t* sidx2;
  const float* sp2;
  // MN-major operands whose tensor map is the 3-D view {64, K rows, MN / 64}:
  // the tile's 64-column blocks arrive in one copy instead of one per block
  int a_mn3d, b_mn3d;
};

__device__ __forceinline__ void decode_tile(const GemmParams& P, int tile, int& m, int& n, int& s) {
  const int mn = P.num_m * P.num_n;
  s = tile / mn;
  const int r = tile - s * mn;
  if (P.m_fast) {
    m = r % P.num_m;
    n = r / P.num_m;
  } else {
    n = r % P.num_n;
    m = r / P.num_n;
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// One 32-column window of this thread's accumulator row, rounded to bf16, into
// the 128 x 64 staging slice `buf` (128-byte rows, 16-byte chunks swizzled by
// row % 8); window c fills the left (c even) or right (c odd) half.
__device__ __forceinline__ void stage_bf16_window(uint32_t buf, int row_in_tile, int c, const float (&g)[32]) {
  const uint32_t row_addr = buf + row_in_tile * 128;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t chunk = static_cast<uint32_t>(((c & 1) << 2) + j) ^ static_cast<uint32_t>(row_in_tile & 7);
    st_shared_v4_b32(row_addr + (chunk << 4), pack_bf16x2(g[8 * j + 0], g[8 * j + 1]),
                     pack_bf16x2(g[8 * j + 2], g[8 * j + 3]), pack_bf16x2(g[8 * j + 4], g[8 * j + 5]),
                     pack_bf16x2(g[8 * j + 6], g[8 * j + 7]));
  }
}

template <bool PAIR>
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* tm, int x, int y, uint32_t bar) {
  if constexpr (PAIR) tma_load_2d_pair(dst, tm, x, y, bar);
  else tma_load_2d(dst, tm, x, y, bar);
}

// An MN-major tile of `cols` (128 or 256) columns starting at column mn (a
// multiple of 64) and 64 k-rows starting at k: one 3-D copy when the map is
// the 3-D view, else one 2-D copy per 64-column block (8 KB apart in shared
// memory, the layout the 3-D copy produces too).
template <bool PAIR>
__device__ __forceinline__ void load_tile_mn(uint32_t dst, const CUtensorMap* tm, bool view3d, int mn, int k, int cols,
                                             uint32_t bar) {
  if (view3d) {
    if constexpr (PAIR) tma_load_3d_pair(dst, tm, 0, k, mn >> 6, bar);
    else tma_load_3d(dst, tm, 0, k, mn >> 6, bar);
  } else {
    for (int j = 0; j < cols / 64; ++j) load_tile<PAIR>(dst + j * 8192, tm, mn + j * 64, k, bar);
  }
}

// MMA completion -> mbarrier at offset `bar`: this CTA's (single form) or both
// CTAs' of the pair (mask 0b11), or the leader's only (mask 0b01).
template <bool PAIR>
__device__ __forceinline__ void mma_commit(uint32_t bar, uint16_t pair_mask) {
  if constexpr (PAIR) umma_commit_pair_mc(bar, pair_mask);
  else umma_commit(bar);
}

template <int EPI, bool A_MN, bool B_MN, bool PAIR>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    kd_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmD, const GemmParams P) {
  using Cfg = GemmCfg<PAIR>;
  constexpr int NST = Cfg::NSTAGE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* staging = smem + NST * Cfg::STAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging + staging_bytes(EPI));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * NST + 7);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile uint32_t* peer_issued = reinterpret_cast<volatile uint32_t*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA rank within the pair (0 = leader: issues the MMAs, owns D rows 0-127 of each tile)
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t bar0 = smem_u32(bars);
  // barrier map: full[s], empty[s], tmem_full[2], tmem_empty[2], drain, and for a
  // pair's wind-down: peer_done (leader: the peer reported its loads), drained
  // (peer: the leader saw every load land)
  const uint32_t full0 = bar0, empty0 = bar0 + 8u * NST;
  const uint32_t tfull0 = bar0 + 16u * NST, tempty0 = tfull0 + 16u;
  const uint32_t drain_bar = tempty0 + 16u;
  const uint32_t peer_done_bar = drain_bar + 8u, drained_bar = drain_bar + 16u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8u * a, 1);
      mbar_init(tempty0 + 8u * a, EPI_WARPS * Cfg::NCTA);  // both CTAs' epilogue warps release
    }
    mbar_init(drain_bar, 1);
    mbar_init(peer_done_bar, 1);
    mbar_init(drained_bar, 1);
    *abort_flag = 0;
    *peer_issued = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if constexpr (EPI != EPI_FWD) prefetch_tmap(&tmD);
  }
  if (warp == 1) {
    tmem_alloc<PAIR>(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish<PAIR>();
    tc_fence_before();
  }
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // the peer's barriers exist before anything signals them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const WaitCtl wc{P.wait_limit_ns, abort_flag, P.status, KD_ERR_TIMEOUT};
  const int num_tiles = P.num_m * P.num_n * P.num_s;
  const int tile0 = PAIR ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
  const int tile_step = PAIR ? static_cast<int>(cluster_count_x()) : static_cast<int>(gridDim.x);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;  // k-blocks whose loads this CTA issued; k-block n uses stage n % NST
      bool ok = true;
      for (int tile = tile0; tile < num_tiles && ok; tile += tile_step) {
        int m, n, s;
        decode_tile(P, tile, m, n, s);
        const int kb0 = s * P.kb_per_split;
        const int kb1 = min(P.kb_total, kb0 + P.kb_per_split);
        // the next chunk's rows (a merged launch)
        const bool next_part = (EPI == EPI_GF || EPI == EPI_FWD_E) && P.m_split > 0 && m >= P.m_split;
        const int a_row = (next_part ? P.a_mn0_2 + (m - P.m_split) * Cfg::TILE_M : P.a_mn0 + m * Cfg::TILE_M) +
                          static_cast<int>(rank) * BM;
        const int b_row = P.b_mn0 + n * BN + static_cast<int>(rank) * Cfg::B_ROWS;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(empty0 + 8u * stage, phase ^ 1u, wc)) {
            ok = false;
            break;
          }
          const uint32_t fb_local = full0 + 8u * stage;
          // the pair's loads all complete on the leader's barrier
          const uint32_t fb = PAIR ? mapa_shared(fb_local, 0) : fb_local;
          const uint32_t a_dst = smem_base + stage * Cfg::STAGE;
          const uint32_t b_dst = a_dst + A_STAGE_BYTES;
          if (!P.debug_withhold_loads) {
            if (leader) mbar_arrive_expect_tx(fb_local, Cfg::NCTA * Cfg::STAGE);
            if (!A_MN) load_tile<PAIR>(a_dst, &tmA, P.a_k0 + kb * BK, a_row, fb);
            else load_tile_mn<PAIR>(a_dst, &tmA, P.a_mn3d != 0, a_row, P.a_k0 + kb * BK, BM, fb);
            if (!B_MN) load_tile<PAIR>(b_dst, &tmB, P.b_k0 + kb * BK, b_row, fb);
            else load_tile_mn<PAIR>(b_dst, &tmB, P.b_mn3d != 0, b_row, P.b_k0 + kb * BK, Cfg::B_ROWS, fb);
            ++issued;
          }
          if (++stage == NST) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Wind-down: no copy may still be in flight when the CTA (or pair) exits.
      // Every k-block older than the last NST was consumed by the MMA (its
      // stage was reused), so only the last NST can be outstanding, and they
      // are outstanding only after an abort.  A pair's loads all signal the
      // leader's barriers, which the peer cannot wait on: the peer reports how
      // many k-blocks it loaded, the leader balances the barriers of k-blocks
      // that only one CTA loaded (arming those only the peer loaded, and
      // completing the peer's share of those only the leader loaded), waits
      // for them to land, and then tells the peer.  Every wait is bounded.
      if constexpr (PAIR) {
        if (!leader) {
          st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<uint32_t*>(peer_issued)), 0), issued);
          mbar_arrive_cluster(mapa_shared(peer_done_bar, 0));
          mbar_wait_quiet(drained_bar, 0, P.wait_limit_ns);
        } else {
          // the peer reaches this point within one wait limit of the leader
          const uint32_t np = mbar_wait_quiet_cluster(peer_done_bar, 0, 2 * P.wait_limit_ns) ? *peer_issued
                                                                                             : issued;
          const uint32_t hi = max(issued, np);
          const uint32_t lo = hi > static_cast<uint32_t>(NST) ? hi - NST : 0u;
          for (uint32_t q = lo; q < hi; ++q) {
            const uint32_t fb = full0 + 8u * (q % NST);
            if (q >= issued) mbar_arrive_expect_tx(fb, Cfg::STAGE);  // only the peer's share was loaded
            else if (q >= np) mbar_complete_tx(fb, Cfg::STAGE);      // the peer's share never will be
          }
          for (uint32_t q = lo; q < hi; ++q)
            mbar_wait_quiet(full0 + 8u * (q % NST), (q / NST) & 1u, P.wait_limit_ns);
          mbar_arrive_cluster(mapa_shared(drained_bar, 1));
        }
      } else if (!ok) {
        const uint32_t lo = issued > static_cast<uint32_t>(NST) ? issued - NST : 0u;
        for (uint32_t q = lo; q < issued; ++q)
          mbar_wait_quiet(full0 + 8u * (q % NST), (q / NST) & 1u, P.wait_limit_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (the leader's, for a pair)
    if (lane == 0 && leader) {
      constexpr uint32_t IDESC = idesc_bf16_f32(Cfg::TILE_M, BN, A_MN, B_MN);
      int stage = 0, local = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = tile0; tile < num_tiles && ok; tile += tile_step, ++local) {
        int m, n, s;
        decode_tile(P, tile, m, n, s);
        const int kb0 = s * P.kb_per_split;
        const int kb1 = min(P.kb_total, kb0 + P.kb_per_split);
        const int acc = local & 1;
        const uint32_t acc_par = (local >> 1) & 1;
        if (!mbar_wait(tempty0 + 8u * acc, acc_par ^ 1u, wc)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(full0 + 8u * stage, phase, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_base + stage * Cfg::STAGE;
          const uint32_t b_base = a_base + A_STAGE_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = A_MN ? sdesc_sw128(a_base + kk * 2048, 8192, 1024)
                                     : sdesc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? sdesc_sw128(b_base + kk * 2048, 8192, 1024)
                                     : sdesc_sw128(b_base + kk * 32, 16, 1024);
            const uint32_t accum = (kb > kb0 || kk > 0) ? 1u : 0u;
            if constexpr (PAIR) umma_bf16_pair(d_tmem, ad, bd, IDESC, accum);
            else umma_bf16(d_tmem, ad, bd, IDESC, accum);
          }
          mma_commit<PAIR>(empty0 + 8u * stage, 0x3);  // frees the stage (in both CTAs) once these MMAs finish
          if (++stage == NST) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit<PAIR>(tfull0 + 8u * acc, 0x3);  // accumulator ready for the epilogue(s)
      }
      // every MMA issued above must be complete before tensor memory is freed
      mma_commit<PAIR>(drain_bar, 0x1);
      mbar_wait_quiet(drain_bar, 0, P.wait_limit_ns);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row_in_tile = q * 32 + lane;
    const bool out_leader = threadIdx.x == 2 * 32;  // issues the epilogue's TMA stores
    const uint32_t staging_base = smem_u32(staging);
    uint32_t slice = 0;  // running count of output slices (alternates staging buffers)
    int local = 0;
    for (int tile = tile0; tile < num_tiles; tile += tile_step, ++local) {
      int m, n, s;
      decode_tile(P, tile, m, n, s);
      const int acc = local & 1;
      const uint32_t acc_par = (local >> 1) & 1;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      // which epilogue this tile runs: the forward statistics or G (runtime only for EPI_GF)
      const bool next_part = (EPI == EPI_GF || EPI == EPI_FWD_E) && P.m_split > 0 && m >= P.m_split;
      const bool is_fwd = EPI == EPI_FWD || next_part;
      const int mm = next_part ? m - P.m_split : m;                         // tile row within its chunk
      const int row0 = mm * Cfg::TILE_M + static_cast<int>(rank) * BM;  // first row of D this CTA holds
      const int r = row0 + row_in_tile;

      // per-row set-up, overlapping the mainloop of this tile
      const int32_t* ids = nullptr;
      const float* ps = nullptr;
      int cur = 0, cid = INT_MAX;
      float cp = 0.f, Mr = 0.f, nl2 = 0.f;
      bool rv = false;
      if constexpr (EPI == EPI_FWD || EPI == EPI_G || EPI == EPI_FWD_E || EPI == EPI_GF) {
        rv = r < (next_part ? P.rows_valid2 : P.rows_valid);
        const int n0 = n * BN;
        ids = (next_part ? P.sidx2 : P.sidx) + static_cast<size_t>(r) * P.K;
        ps = (next_part ? P.sp2 : P.sp) + static_cast<size_t>(r) * P.K;
        int lo = 0, hi = P.K;  // first sorted position with id >= n0
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (__ldg(ids + mid) < n0) lo = mid + 1;
          else hi = mid;
        }
        cur = lo;
        if (cur < P.K) {
          cid = __ldg(ids + cur);
          cp = __ldg(ps + cur);
        }
        if constexpr (EPI == EPI_G || EPI == EPI_GF) {
          if (!is_fwd && rv) {
            Mr = __ldg(P.rowM + r);
            nl2 = -__ldg(P.lse + r) * kLog2e;
          }
        }
      }

      bool ok = mbar_wait(tfull0 + 8u * acc, acc_par, wc);
      // all four epilogue warps must take the same decision: the TMA-store
      // paths synchronise them on a named barrier below
      if constexpr (EPI != EPI_FWD) ok = named_bar_and(EPI_BAR_ID, EPI_WARPS * 32, ok);
      else ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();

      float run_m = -INFINITY, run_s = 0.f, pz = 0.f;
      if constexpr (EPI == EPI_FWD_E) {
        // first pass over the accumulator: the row's maximum over the tile's
        // vocabulary columns, the reference point of the kept exponentials
        float tmax = -INFINITY;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld32(taddr + c * 32, v);
          const int nv = P.V - (n * BN + c * 32);  // <= 0 past the vocabulary
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < nv) tmax = fmaxf(tmax, v[j]);
        }
        run_m = tmax * kLog2e;
      }
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        float v[32];
        tmem_ld32(taddr + c * 32, v);
        const int col0 = n * BN + c * 32;
        if (EPI == EPI_FWD || (EPI == EPI_GF && is_fwd)) {
          if (col0 < P.V) {
            const int nv = min(32, P.V - col0);
            float wm = -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j < nv) wm = fmaxf(wm, v[j]);
            const float m_new = fmaxf(run_m, wm * kLog2e);
            float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              if (j + 0 < nv) s0 += ex2(fmaf(v[j + 0], kLog2e, -m_new));
              if (j + 1 < nv) s1 += ex2(fmaf(v[j + 1], kLog2e, -m_new));
              if (j + 2 < nv) s2 += ex2(fmaf(v[j + 2], kLog2e, -m_new));
              if (j + 3 < nv) s3 += ex2(fmaf(v[j + 3], kLog2e, -m_new));
            }
            run_s = run_s * ex2(run_m - m_new) + ((s0 + s1) + (s2 + s3));
            run_m = m_new;
            while (cid < col0 + 32) {
              const int off = cid - col0;
              float sel = 0.f;
#pragma unroll
              for (int j = 0; j < 32; ++j) sel = (j == off) ? v[j] : sel;
              pz = fmaf(cp, sel, pz);
              ++cur;
              cid = cur < P.K ? __ldg(ids + cur) : INT_MAX;
              cp = cur < P.K ? __ldg(ps + cur) : 0.f;
            }
          }
        } else if (EPI == EPI_G || EPI == EPI_GF) {
          // two 32-column windows fill one 128 x 64 bf16 slice of the staging buffer
          const uint32_t buf = staging_base + (slice & 1u) * OUT_SLICE_BYTES;
          if ((c & 1) == 0) {
            if (out_leader) bulk_wait_read1();  // the store that last read `buf` is done with it
            named_bar_sync(EPI_BAR_ID, EPI_WARPS * 32);
          }
          float g[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) g[j] = rv ? Mr * ex2(fmaf(v[j], kLog2e, nl2)) : 0.f;
          while (cid < col0 + 32) {
            const int off = cid - col0;
#pragma unroll
            for (int j = 0; j < 32; ++j) g[j] = (j == off) ? g[j] - cp : g[j];
            ++cur;
            cid = cur < P.K ? __ldg(ids + cur) : INT_MAX;
            cp = cur < P.K ? __ldg(ps + cur) : 0.f;
          }
          stage_bf16_window(buf, row_in_tile, c, g);
          if (c & 1) {
            fence_proxy_async_smem();
            named_bar_sync(EPI_BAR_ID, EPI_WARPS * 32);
            if (out_leader) {
              tma_store_2d(&tmD, n * BN + (c >> 1) * G_SLICE_COLS, P.out_row0 + row0, buf);
              bulk_commit();
            }
            ++slice;
          }
        } else if (EPI == EPI_FWD_E) {
          const uint32_t buf = staging_base + (slice & 1u) * OUT_SLICE_BYTES;
          if ((c & 1) == 0) {
            if (out_leader) bulk_wait_read1();  // the store that last read `buf` is done with it
            named_bar_sync(EPI_BAR_ID, EPI_WARPS * 32);
          }
          const int nv = P.V - col0;  // <= 0 past the vocabulary
          float e[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) e[j] = (j < nv) ? ex2(fmaf(v[j], kLog2e, -run_m)) : 0.f;
          float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            s0 += e[j];
            s1 += e[j + 1];
            s2 += e[j + 2];
            s3 += e[j + 3];
          }
          run_s += (s0 + s1) + (s2 + s3);
          while (cid < col0 + 32) {
            const int off = cid - col0;
            float sel = 0.f;
#pragma unroll
            for (int j = 0; j < 32; ++j) sel = (j == off) ? v[j] : sel;
            pz = fmaf(cp, sel, pz);
            ++cur;
            cid = cur < P.K ? __ldg(ids + cur) : INT_MAX;
            cp = cur < P.K ? __ldg(ps + cur) : 0.f;
          }
          if (!rv) {
#pragma unroll
            for (int j = 0; j < 32; ++j) e[j] = 0.f;
          }
          stage_bf16_window(buf, row_in_tile, c, e);
          if (c & 1) {
            fence_proxy_async_smem();
            named_bar_sync(EPI_BAR_ID, EPI_WARPS * 32);
            if (out_leader) {
              tma_store_2d(&tmD, n * BN + (c >> 1) * G_SLICE_COLS, (next_part ? P.out_row0_2 : P.out_row0) + row0, buf);
              bulk_commit();
            }
            ++slice;
          }
        } else {  // EPI_F32
          const uint32_t buf = staging_base + (slice & 1u) * OUT_SLICE_BYTES;
          if (out_leader) bulk_wait_read1();  // the store that last read `buf` is done with it
          named_bar_sync(EPI_BAR_ID, EPI_WARPS * 32);
          const uint32_t row_addr = buf + row_in_tile * 128;
#pragma unroll
          for (int j = 0; j < 8; ++j)  // 16-byte chunk j of the row goes to chunk j ^ (row % 8)
            st_shared_v4(row_addr + ((j ^ (row_in_tile & 7)) << 4), v[4 * j] * P.scale,
                         v[4 * j + 1] * P.scale, v[4 * j + 2] * P.scale, v[4 * j + 3] * P.scale);
          fence_proxy_async_smem();
          named_bar_sync(EPI_BAR_ID, EPI_WARPS * 32);
          if (out_leader) {
            const int y = P.out_row0 + s * P.split_rows + row0;
            if (P.reduce_add) tma_reduce_add_2d(&tmD, col0, y, buf);
            else tma_store_2d(&tmD, col0, y, buf);
            bulk_commit();
          }
          ++slice;
        }
      }
      // release the accumulator buffer to the MMA warp (the leader's, for a pair)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR && !leader) mbar_arrive_cluster(mapa_shared(tempty0 + 8u * acc, 0));
        else mbar_arrive(tempty0 + 8u * acc);
      }
      if constexpr (EPI == EPI_FWD || EPI == EPI_FWD_E || EPI == EPI_GF) {
        if (rv && (EPI != EPI_GF || is_fwd)) {
          const size_t o = static_cast<size_t>(n) * P.ld_part + r + (EPI == EPI_FWD_E && next_part ? P.part_row2 : 0);
          P.part_m[o] = run_m;
          P.part_s[o] = run_s;
          P.part_pz[o] = pz;
        }
      }
    }
  }

  if constexpr (EPI != EPI_FWD) {
    if (threadIdx.x == 2 * 32) bulk_wait0();  // output stores complete before the CTA exits
  }
  __syncthreads();
  // a pair stays resident until neither CTA touches the other's memory any more
  if constexpr (PAIR) cluster_sync();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc<PAIR>(tmem_base, TMEM_COLS);
  }
}

}  // namespace kd
