// Host side of the C ABI declared in include/kdtopk.h: argument checks,
// workspace carving, TMA descriptor set-up and the chunk loop on the caller's
// stream.  Method: fused, chunked top-K KL distillation loss ("Efficient
// Knowledge Distillation for LLMs: Offline Top-K Logits and a Fused Chunked KL
// Loss"; aimodeling.com "Second cut", thorstenmeyerai.com pipeline steps
// "Train in chunks" / "Recompute backward").
//
// Per chunk of `chunk` token rows:
//   prep      ids sorted per row, M_t, E_t, id range check
//   forward   logits GEMM with fused online softmax partials + top-K gather
//             (logits stay in tensor memory), combine -> lse_t, L_t, loss
//   backward  logits GEMM again with G = M softmax - p formed in the epilogue
//             (bf16 [chunk, V] operand), dH = G W (split-K, then a reduction),
//             dW += G^T H (fp32 read-modify-write of the caller's dW)
// The fused step is pipelined by one chunk: chunk c's G GEMM and chunk c+1's
// forward GEMM run as one launch over both chunks' rows (they share every W
// tile).  The no-recompute fused step keeps the forward's tile-normalised
// exponentials in the G buffer and forms G from them elementwise once lse is
// known, so the backward starts at dH.  The teacher-cache builder (top-K ids
// and probabilities of teacher logits) and a gradient scale-and-round helper
// complete the ABI.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <type_traits>
#include <vector>

#include "kd_aux.cuh"
#include "kd_cache.cuh"
#include "kd_gemm.cuh"
#include "kdtopk.h"

namespace {

using namespace kd;

// ------------------------------------------------------------------ helpers
size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2-D bf16 tensor map, 128-byte swizzle, zero fill out of bounds.
bool tmap_bf16(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
               uint32_t box_inner, uint32_t box_outer) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D view {64, rows, mn / 64} of a row-major bf16 matrix [rows, mn] read as an
// MN-major GEMM operand (mn the contiguous index): one box of {64, BK, nblk}
// is nblk consecutive 64-column blocks of BK rows, laid out in shared memory
// exactly as nblk 2-D boxes of {64, BK}.  Only when mn % 64 == 0, so that the
// view never reaches past a row's last element; out-of-range rows and blocks
// are zero-filled as in the 2-D map.
bool tmap_bf16_mn3d(CUtensorMap* tm, const void* base, uint64_t mn, uint64_t rows, uint64_t row_bytes,
                    uint32_t nblk) {
  auto enc = encode_fn();
  if (!enc || mn % 64 != 0) return false;
  cuuint64_t dims[3] = {64, rows, mn / 64};
  cuuint64_t strides[2] = {row_bytes, 128};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(BK), nblk};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// An MN-major operand's map: the 3-D view when mn allows it (*view3d = 1),
// else the 2-D map with 64-column boxes.
bool tmap_bf16_mn(CUtensorMap* tm, int* view3d, const void* base, uint64_t mn, uint64_t rows, uint64_t row_bytes,
                  uint32_t tile_cols) {
  *view3d = 0;
  if (mn % 64 == 0 && tmap_bf16_mn3d(tm, base, mn, rows, row_bytes, tile_cols / 64)) {
    *view3d = 1;
    return true;
  }
  return tmap_bf16(tm, base, mn, rows, row_bytes, 64, BK);
}

// 2-D fp32 tensor map for the GEMM outputs: 32-column x 128-row boxes, 128-byte swizzle.
bool tmap_f32_out(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(OUT_SLICE_COLS), static_cast<cuuint32_t>(BM)};
  cuuint32_t estr[2] = {1, 1};
  return enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int current_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 148;
  }
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 148;
  }
  return n;
}

// The kernels are built for sm_103a only.
bool device_supported() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return false;
  return major == 10 && minor == 3;
}

// Rows of G that one dW = G^T H launch reduces over.  A dW tile's mainloop is
// only K = chunk rows long while its epilogue read-modify-writes a 128 x 256
// fp32 tile of dW, so for short chunks the epilogue cannot hide behind the
// tensor cores; grouping consecutive chunks (G kept for the whole group)
// lengthens K and divides dW's HBM traffic per chunk.  KD_DW_GROUP_ROWS
// overrides the default 4096 rows (at most 4 chunks; 0 or fewer rows than two
// chunks: no grouping).
int dw_group_rows() {
  static int v = [] {
    const char* e = std::getenv("KD_DW_GROUP_ROWS");
    return e ? std::atoi(e) : 4096;
  }();
  return v;
}

// CTA-pair (two-CTA cluster, 256-row tile) GEMMs for chunks of at least 256
// rows; KD_PAIR=0 (read once per process) selects the single-CTA form.
bool pair_enabled() {
  static bool v = [] {
    const char* e = std::getenv("KD_PAIR");
    return !(e && std::atoi(e) == 0);
  }();
  return v;
}

// The fused steps run two chunks' projections as one launch (chunk c's G GEMM
// with chunk c+1's forward, or without the recompute the forward GEMMs of
// chunks c and c+1); KD_MERGE_LOGITS=0 (read once per process) keeps them apart.
bool merge_enabled() {
  static bool v = [] {
    const char* e = std::getenv("KD_MERGE_LOGITS");
    return !(e && std::atoi(e) == 0);
  }();
  return v;
}

uint64_t wait_limit_ns() {
  static uint64_t v = [] {
    const char* e = std::getenv("KD_WAIT_LIMIT_MS");
    long ms = e ? std::atol(e) : 0;
    if (ms <= 0) ms = 4000;
    return static_cast<uint64_t>(ms) * 1000000ull;
  }();
  return v;
}

// ------------------------------------------------------------------ profiler
struct Profiler {
  bool on = false;
  std::vector<cudaEvent_t> ev;      // pairs (start, stop)
  std::vector<int> kind;            // per pair
  size_t used = 0;
  int64_t dropped = 0;
  static constexpr size_t kPairs = 16384;
};
Profiler g_prof;

int prof_begin(int k, cudaStream_t st) {
  if (!g_prof.on || g_prof.used >= g_prof.kind.size()) {
    if (g_prof.on) ++g_prof.dropped;
    return -1;
  }
  const int slot = static_cast<int>(g_prof.used++);
  g_prof.kind[slot] = k;
  cudaEventRecord(g_prof.ev[2 * slot], st);
  return slot;
}
void prof_end(int slot, cudaStream_t st) {
  if (slot >= 0) cudaEventRecord(g_prof.ev[2 * slot + 1], st);
}

// ------------------------------------------------------------------ plan
struct Plan {
  int64_t T;
  int d, V, K, C, Cpad, Kpad, nt, S, kbps_dh, nchunks;
  int prep_bufs;  // sorted-cache buffers: 2 when one chunk's backward overlaps the next chunk's forward
  size_t prep_stride;  // bytes between them
  bool pair;     // chunk GEMMs run as CTA pairs (tiles of 256 rows)
  int tile_m;    // rows per GEMM tile: 256 for pairs, 128 otherwise
  int dw_group;  // chunks whose G rows one dW GEMM consumes (K = dw_group * C)
  int64_t ldg;
  // leading dimension of the softmax partials: two chunks' rows when the
  // no-recompute step can run two chunks' forward GEMMs as one launch
  int part_ld;
  size_t off_status, off_sidx, off_sp, off_M, off_E, off_pm, off_ps, off_pz, off_Lrow, off_G, off_dhp, total;
};

// Split of the dH = G W reduction over V so that (row tiles x d tiles x
// splits) fills the SMs with few partial waves.
int choose_splits(int64_t mn_tiles, int64_t kb_total, int sms) {
  int best = 1;
  double best_eff = 0.0;
  for (int s = 1; s <= 8; ++s) {
    if (kb_total / s < 4) break;
    const int64_t units = mn_tiles * s;
    const int64_t waves = ceil_div(units, sms);
    const double eff = static_cast<double>(units) / static_cast<double>(waves * sms);
    if (eff > best_eff + 0.02) {
      best = s;
      best_eff = eff;
    }
  }
  return best;
}

kd_status make_plan(int64_t T, int d, int V, int K, int chunk, int what, Plan* pl) {
  if (T < 1 || d < 1 || V < 1 || K < 1 || chunk < 1 || (what & KD_WS_FUSED) == 0) return KD_ERR_INVALID_ARG;
  if (K > V) return KD_ERR_INVALID_ARG;
  if (d % 8 != 0 || K > 1024) return KD_ERR_UNSUPPORTED;
  if (T > (int64_t(1) << 31) - 256 || static_cast<int64_t>(V) * d >= (int64_t(1) << 40)) return KD_ERR_UNSUPPORTED;
  Plan& p = *pl;
  p.T = T;
  p.d = d;
  p.V = V;
  p.K = K;
  p.C = static_cast<int>(std::min<int64_t>(chunk, T));
  p.pair = pair_enabled() && align_up(p.C, BM) >= 2 * BM;
  p.tile_m = p.pair ? 2 * BM : BM;
  p.Cpad = static_cast<int>(align_up(p.C, p.tile_m));
  p.Kpad = 32;
  while (p.Kpad < K) p.Kpad <<= 1;
  p.nt = static_cast<int>(ceil_div(V, BN));
  p.ldg = static_cast<int64_t>(align_up(V, 8));
  p.nchunks = static_cast<int>(ceil_div(T, p.C));
  // grouping needs the chunks' G rows to line up with H rows: chunk == Cpad
  p.dw_group = (p.C == p.Cpad) ? std::min(4, std::max(1, dw_group_rows() / p.C)) : 1;
  p.dw_group = std::min(p.dw_group, p.nchunks);
  const int64_t kb_v = ceil_div(V, BK);
  const int sms = current_sm_count();
  int S = choose_splits(static_cast<int64_t>(p.Cpad / p.tile_m) * ceil_div(d, BN), kb_v, p.pair ? sms / 2 : sms);
  p.kbps_dh = static_cast<int>(ceil_div(kb_v, S));
  p.S = static_cast<int>(ceil_div(kb_v, p.kbps_dh));
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  p.off_status = take(256);  // int status + double loss accumulator
  // prep outputs (sorted ids, their p, M_t, E_t); the fused step keeps two sets
  p.prep_bufs = ((what & KD_WS_FUSED) == KD_WS_FUSED) ? 2 : 1;
  const size_t prep_start = o;
  p.off_sidx = take(size_t(p.Cpad) * K * 4);
  p.off_sp = take(size_t(p.Cpad) * K * 4);
  p.off_M = take(size_t(p.Cpad) * 4);
  p.off_E = take(size_t(p.Cpad) * 4);
  p.prep_stride = o - prep_start;
  if (p.prep_bufs == 2) o += p.prep_stride;
  p.off_pm = p.off_ps = p.off_pz = p.off_Lrow = 0;
  p.off_G = p.off_dhp = 0;
  p.part_ld = ((what & KD_WS_FUSED) == KD_WS_FUSED && p.dw_group % 2 == 0) ? 2 * p.Cpad : p.Cpad;
  if (what & KD_WS_FORWARD) {
    p.off_pm = take(size_t(p.nt) * p.part_ld * 4);
    p.off_ps = take(size_t(p.nt) * p.part_ld * 4);
    p.off_pz = take(size_t(p.nt) * p.part_ld * 4);
    p.off_Lrow = take(size_t(p.Cpad) * 8);
  }
  if (what & KD_WS_BACKWARD) {
    p.off_G = take(size_t(p.dw_group) * p.Cpad * p.ldg * 2);
    p.off_dhp = take(size_t(p.S) * p.Cpad * d * 4);
  }
  p.total = o;
  return KD_OK;
}

// Persistent launch: one CTA (or CTA pair) per SM, at most one per tile.
template <int EPI, bool A_MN, bool B_MN, bool PAIR>
cudaError_t launch_gemm(int kind, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& td,
                        const GemmParams& P, int sms, cudaStream_t st) {
  auto kern = kd_gemm_kernel<EPI, A_MN, B_MN, PAIR>;
  constexpr size_t smem = gemm_smem_bytes<PAIR>(EPI);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int64_t tiles = static_cast<int64_t>(P.num_m) * P.num_n * P.num_s;
  const int slot = prof_begin(kind, st);
  if constexpr (PAIR) {
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.blockDim = dim3(GEMM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // pairs that can be resident at once (clusters sit within one GPC), asked once per kernel
    static std::atomic<int> resident{0};
    int res = resident.load(std::memory_order_relaxed);
    if (res == 0) {
      cfg.gridDim = dim3(static_cast<unsigned>(std::max(2, sms)));
      if (cudaOccupancyMaxActiveClusters(&res, kern, &cfg) != cudaSuccess || res <= 0) {
        cudaGetLastError();
        res = std::max(1, sms / 2);
      }
      resident.store(res, std::memory_order_relaxed);
    }
    const int pairs = static_cast<int>(std::min<int64_t>(tiles, std::min(res, std::max(1, sms / 2))));
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
    e = cudaLaunchKernelEx(&cfg, kern, ta, tb, td, P);
  } else {
    const int grid = static_cast<int>(std::min<int64_t>(tiles, sms));
    kern<<<grid, GEMM_THREADS, smem, st>>>(ta, tb, td, P);
    e = cudaGetLastError();
  }
  prof_end(slot, st);
  return e;
}

// Dispatch on the pair form chosen at run time.
template <int EPI, bool A_MN, bool B_MN>
cudaError_t launch_gemm_any(bool pair, int kind, const CUtensorMap& ta, const CUtensorMap& tb,
                            const CUtensorMap& td, const GemmParams& P, int sms, cudaStream_t st) {
  return pair ? launch_gemm<EPI, A_MN, B_MN, true>(kind, ta, tb, td, P, sms, st)
              : launch_gemm<EPI, A_MN, B_MN, false>(kind, ta, tb, td, P, sms, st);
}

GemmParams base_params(int* status) {
  GemmParams P;
  std::memset(&P, 0, sizeof(P));
  P.num_s = 1;
  P.m_fast = 1;
  P.wait_limit_ns = wait_limit_ns();
  P.status = status;
  P.scale = 1.f;
  return P;
}

// MODE_KEEP (with MODE_FWD | MODE_BWD): the forward GEMM keeps the chunk's
// tile-normalised exponentials in the G buffer and an elementwise pass turns
// them into G, instead of recomputing the logits in the backward.
enum { MODE_FWD = 1, MODE_BWD = 2, MODE_KEEP = 4 };

kd_status run(int mode, const void* H, const void* W, const int32_t* idx, const float* p, const float* lse_in,
              int64_t T, int d, int V, int K, int chunk, float dloss, float* loss, float* lse, float* loss_rows,
              float* dH, float* dW, int accumulate, void* ws, size_t ws_bytes, cudaStream_t st) {
  if (!H || !W || !idx || !p || !ws) return KD_ERR_INVALID_ARG;
  if ((mode & MODE_FWD) && (!loss || !lse)) return KD_ERR_INVALID_ARG;
  if ((mode & MODE_BWD) && (!dH || !dW)) return KD_ERR_INVALID_ARG;
  if (mode == MODE_BWD && !lse_in) return KD_ERR_INVALID_ARG;
  Plan pl;
  const int what = (mode & MODE_FWD ? KD_WS_FORWARD : 0) | (mode & MODE_BWD ? KD_WS_BACKWARD : 0);
  kd_status rc = make_plan(T, d, V, K, chunk, what, &pl);
  if (rc != KD_OK) return rc;
  if (!aligned16(H) || !aligned16(W) || (reinterpret_cast<uintptr_t>(ws) & 255u) ||
      (reinterpret_cast<uintptr_t>(idx) & 3u) || (reinterpret_cast<uintptr_t>(p) & 3u) ||
      (dH && !aligned16(dH)) || (dW && !aligned16(dW)))
    return KD_ERR_UNSUPPORTED;
  if (ws_bytes < pl.total) return KD_ERR_WORKSPACE;
  if (!device_supported()) return KD_ERR_UNSUPPORTED;
  if (!encode_fn()) return KD_ERR_CUDA;
  const int sms = current_sm_count();

  uint8_t* w8 = static_cast<uint8_t*>(ws);
  int* status = reinterpret_cast<int*>(w8 + pl.off_status);
  double* loss_acc = reinterpret_cast<double*>(w8 + pl.off_status + 8);
  float* pm = reinterpret_cast<float*>(w8 + pl.off_pm);
  float* ps = reinterpret_cast<float*>(w8 + pl.off_ps);
  float* ppz = reinterpret_cast<float*>(w8 + pl.off_pz);
  double* Lrow = reinterpret_cast<double*>(w8 + pl.off_Lrow);
  __nv_bfloat16* G = reinterpret_cast<__nv_bfloat16*>(w8 + pl.off_G);
  float* dhp = reinterpret_cast<float*>(w8 + pl.off_dhp);

  // TMA descriptors (all bf16, 128-byte swizzle, 64-element inner boxes)
  CUtensorMap tmH_k, tmW_k, tmG_k, tmW_mn, tmG_mn, tmH_mn, tmDhp, tmDW;
  int w_mn3d = 0, g_mn3d = 0, h_mn3d = 0;  // MN-major maps that are 3-D views
  const uint64_t hrow = uint64_t(d) * 2;
  const bool pr = pl.pair;
  // K-major B (W in the logits GEMMs): each CTA of a pair stages half of the 256 columns
  bool ok = tmap_bf16(&tmH_k, H, d, T, hrow, BK, BM) && tmap_bf16(&tmW_k, W, d, V, hrow, BK, pr ? BN / 2 : BN);
  if (mode & MODE_BWD) {
    const uint64_t grows = uint64_t(pl.dw_group) * pl.Cpad;  // G rows held in the workspace
    ok = ok && tmap_bf16(&tmG_k, G, V, grows, uint64_t(pl.ldg) * 2, BK, BM) &&
         tmap_bf16_mn(&tmW_mn, &w_mn3d, W, d, V, hrow, pr ? BN / 2 : BN) &&
         tmap_bf16_mn(&tmG_mn, &g_mn3d, G, V, grows, uint64_t(pl.ldg) * 2, BM) &&
         tmap_bf16_mn(&tmH_mn, &h_mn3d, H, d, T, hrow, pr ? BN / 2 : BN) &&
         tmap_f32_out(&tmDhp, dhp, d, uint64_t(pl.S) * pl.Cpad, uint64_t(d) * 4) &&
         tmap_f32_out(&tmDW, dW, d, V, uint64_t(d) * 4);
  }
  if (!ok) return KD_ERR_CUDA;

  if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return KD_ERR_CUDA;

  // rows of the id / probability cache that 16-byte loads can read
  const int vec_rows = (K % 4 == 0 && aligned16(idx) && aligned16(p)) ? 1 : 0;

  const bool keep = (mode & MODE_KEEP) != 0;
  const int kb_d = static_cast<int>(ceil_div(d, BK));
  auto t0_of = [&](int c) { return int64_t(c) * pl.C; };
  auto rows_of = [&](int c) { return static_cast<int>(std::min<int64_t>(pl.C, T - t0_of(c))); };
  auto gslot_of = [&](int c) { return c % pl.dw_group; };  // chunk c's G rows: [gslot * Cpad, +Cpad)
  // the no-recompute step runs chunk pairs (c even, c + 1) through one forward
  // launch when the G slots of a pair are adjacent (an even dW group) and the
  // partials hold two chunks; the pair's second chunk keeps its partials in the
  // second half
  const bool kmerge = keep && (mode & MODE_FWD) && (mode & MODE_BWD) && pl.part_ld == 2 * pl.Cpad &&
                      pl.prep_bufs == 2 && pl.nchunks > 1 && merge_enabled();
  auto part_off = [&](int c) { return (kmerge && (c & 1)) ? size_t(pl.Cpad) : size_t(0); };
  // the sorted cache of chunk c lives in prep buffer c % prep_bufs
  auto pbuf = [&](int c, size_t off) { return w8 + off + size_t(c % pl.prep_bufs) * pl.prep_stride; };
  auto sidx_of = [&](int c) { return reinterpret_cast<int32_t*>(pbuf(c, pl.off_sidx)); };
  auto sp_of = [&](int c) { return reinterpret_cast<float*>(pbuf(c, pl.off_sp)); };
  auto rowM_of = [&](int c) { return reinterpret_cast<float*>(pbuf(c, pl.off_M)); };
  auto rowE_of = [&](int c) { return reinterpret_cast<float*>(pbuf(c, pl.off_E)); };
  auto logits_params = [&](int c) {
    GemmParams L = base_params(status);
    L.num_m = pl.Cpad / pl.tile_m;
    L.num_n = pl.nt;
    L.kb_total = L.kb_per_split = kb_d;
    L.a_mn0 = static_cast<int>(t0_of(c));
    L.rows_valid = rows_of(c);
    L.V = V;
    L.K = K;
    L.sidx = sidx_of(c);
    L.sp = sp_of(c);
    L.part_m = pm;
    L.part_s = ps;
    L.part_pz = ppz;
    L.ld_part = pl.part_ld;
    L.out_row0 = gslot_of(c) * pl.Cpad;
    L.rowM = rowM_of(c);
    L.lse = ((mode & MODE_FWD) ? lse : lse_in) + t0_of(c);
    return L;
  };
  auto check = [&](cudaError_t e) { return e == cudaSuccess; };

  // ---- the steps of one chunk
  auto prep = [&](int c) {
    const int slot = prof_begin(KD_K_PREP, st);
    const unsigned blocks = static_cast<unsigned>(ceil_div(pl.Cpad, PREP_WARPS));
    const int32_t* ic = idx + t0_of(c) * K;
    const float* pc = p + t0_of(c) * K;
#define KD_PREP(EPT)                                                                                          \
  kd_prep_kernel<EPT><<<blocks, PREP_WARPS * 32, 0, st>>>(ic, pc, rows_of(c), pl.Cpad, K, V, vec_rows, sidx_of(c), \
                                                         sp_of(c), rowM_of(c), rowE_of(c), status)
    switch (pl.Kpad) {
      case 32: KD_PREP(1); break;
      case 64: KD_PREP(2); break;
      case 128: KD_PREP(4); break;
      case 256: KD_PREP(8); break;
      case 512: KD_PREP(16); break;
      default: KD_PREP(32); break;  // Kpad 1024 (K <= 1024 is checked)
    }
#undef KD_PREP
    const cudaError_t e = cudaGetLastError();
    prof_end(slot, st);
    return check(e);
  };
  auto forward_gemm = [&](int c) {
    const GemmParams P = logits_params(c);
    if (keep) return check(launch_gemm_any<EPI_FWD_E, false, false>(pr, KD_K_LOGITS_FWD, tmH_k, tmW_k, tmG_k, P, sms, st));
    return check(launch_gemm_any<EPI_FWD, false, false>(pr, KD_K_LOGITS_FWD, tmH_k, tmW_k, tmH_k, P, sms, st));
  };
  auto combine = [&](int c) {
    const int rows = rows_of(c);
    const size_t po = part_off(c);
    const int slot = prof_begin(KD_K_COMBINE, st);
    kd_combine_kernel<<<static_cast<unsigned>(ceil_div(rows, 32)), COMBINE_WARPS * 32, 0, st>>>(
        pm + po, ps + po, ppz + po, pl.nt, pl.part_ld, rows, rowM_of(c), rowE_of(c), lse + t0_of(c),
        loss_rows ? loss_rows + t0_of(c) : nullptr, Lrow);
    kd_loss_reduce_kernel<<<1, 1024, 0, st>>>(Lrow, rows, loss_acc, c == 0 ? 1 : 0,
                                              c == pl.nchunks - 1 ? loss : nullptr);
    cudaError_t e = cudaGetLastError();
    prof_end(slot, st);
    if (e == cudaSuccess && keep) {  // G from the kept exponentials, in place, now that lse is known
      const int gs = prof_begin(KD_K_G_FROM_E, st);
      kd_g_from_e_kernel<<<static_cast<unsigned>(rows), GPASS_THREADS, 0, st>>>(
          G + size_t(gslot_of(c)) * pl.Cpad * pl.ldg, pl.ldg, rows, V, K, sidx_of(c), sp_of(c), rowM_of(c),
          lse + t0_of(c), pm + po, pl.part_ld);
      e = cudaGetLastError();
      prof_end(gs, st);
    }
    return check(e);
  };
  // the no-recompute step: chunks c and c+1's forward GEMMs (kept exponentials)
  // in one launch, sharing every W tile through L2
  auto forward_pair = [&](int c) {
    GemmParams P = logits_params(c);
    const GemmParams F = logits_params(c + 1);
    P.m_split = P.num_m;
    P.num_m = 2 * P.num_m;
    P.a_mn0_2 = F.a_mn0;
    P.rows_valid2 = F.rows_valid;
    P.sidx2 = F.sidx;
    P.sp2 = F.sp;
    P.out_row0_2 = F.out_row0;
    P.part_row2 = pl.Cpad;
    return check(launch_gemm_any<EPI_FWD_E, false, false>(pr, KD_K_LOGITS_FWD, tmH_k, tmW_k, tmG_k, P, sms, st));
  };
  auto g_gemm = [&](int c) {
    const GemmParams P = logits_params(c);
    return check(launch_gemm_any<EPI_G, false, false>(pr, KD_K_LOGITS_G, tmH_k, tmW_k, tmG_k, P, sms, st));
  };
  // chunk c's G and chunk c+1's forward in one launch: both halves share every W tile
  auto g_and_next_forward = [&](int c) {
    GemmParams P = logits_params(c);
    const GemmParams F = logits_params(c + 1);
    P.m_split = P.num_m;
    P.num_m = 2 * P.num_m;
    P.a_mn0_2 = F.a_mn0;
    P.rows_valid2 = F.rows_valid;
    P.sidx2 = F.sidx;
    P.sp2 = F.sp;
    return check(launch_gemm_any<EPI_GF, false, false>(pr, KD_K_LOGITS_GF, tmH_k, tmW_k, tmG_k, P, sms, st));
  };
  auto dh_and_dw = [&](int c) {
    const int gslot = gslot_of(c);
    GemmParams Q = base_params(status);  // dH partials = G W, split over V
    Q.num_m = pl.Cpad / pl.tile_m;
    Q.num_n = static_cast<int>(ceil_div(d, BN));
    Q.num_s = pl.S;
    Q.kb_total = static_cast<int>(ceil_div(V, BK));
    Q.kb_per_split = pl.kbps_dh;
    Q.split_rows = pl.Cpad;
    Q.a_mn0 = gslot * pl.Cpad;
    Q.b_mn3d = w_mn3d;
    if (!check(launch_gemm_any<EPI_F32, false, true>(pr, KD_K_GEMM_DH, tmG_k, tmW_mn, tmDhp, Q, sms, st)))
      return false;
    {
      const int64_t n4 = int64_t(rows_of(c)) * d / 4;
      const int slot = prof_begin(KD_K_DH_REDUCE, st);
      kd_dh_reduce_kernel<<<static_cast<unsigned>(std::min<int64_t>(ceil_div(n4, 256), 4L * sms)), 256, 0, st>>>(
          reinterpret_cast<const float4*>(dhp), pl.S, int64_t(pl.Cpad) * d / 4, n4, dloss,
          reinterpret_cast<float4*>(dH + t0_of(c) * d));
      const cudaError_t e = cudaGetLastError();
      prof_end(slot, st);
      if (e != cudaSuccess) return false;
    }
    if (gslot == pl.dw_group - 1 || c == pl.nchunks - 1) {
      // dW (+)= G^T H over the group's chunks, fp32; the first group stores, the rest add in L2
      const int first = c - gslot;
      GemmParams R = base_params(status);
      R.num_m = static_cast<int>(ceil_div(V, pl.tile_m));
      R.num_n = static_cast<int>(ceil_div(d, BN));
      R.m_fast = 0;
      R.kb_total = R.kb_per_split = (gslot + 1) * pl.Cpad / BK;
      R.b_k0 = static_cast<int>(int64_t(first) * pl.C);
      R.reduce_add = (first == 0 && !accumulate) ? 0 : 1;
      R.scale = dloss;
      R.a_mn3d = g_mn3d;
      R.b_mn3d = h_mn3d;
      if (!check(launch_gemm_any<EPI_F32, true, true>(pr, KD_K_GEMM_DW, tmG_mn, tmH_mn, tmDW, R, sms, st)))
        return false;
    }
    return true;
  };

  const bool fused = (mode & MODE_FWD) && (mode & MODE_BWD);
  if (kmerge) {
    // no-recompute path: the forward GEMMs of chunks c and c+1 (c even) as one
    // launch, then each chunk's combine, G pass and backward GEMMs in order
    for (int c = 0; c < pl.nchunks; c += 2) {
      const bool pair = c + 1 < pl.nchunks;
      if (!prep(c)) return KD_ERR_CUDA;
      if (pair) {
        if (!prep(c + 1) || !forward_pair(c)) return KD_ERR_CUDA;
      } else if (!forward_gemm(c)) {
        return KD_ERR_CUDA;
      }
      if (!combine(c) || (pair && !combine(c + 1))) return KD_ERR_CUDA;
      if (!dh_and_dw(c) || (pair && !dh_and_dw(c + 1))) return KD_ERR_CUDA;
    }
    return KD_OK;
  }
  if (fused && !keep && pl.prep_bufs == 2 && pl.nchunks > 1 && merge_enabled()) {
    // recompute path, software-pipelined by one chunk: after chunk c's forward and
    // combine, chunk c's G GEMM runs together with chunk c+1's forward GEMM
    if (!prep(0) || !forward_gemm(0) || !combine(0)) return KD_ERR_CUDA;
    for (int c = 0; c < pl.nchunks; ++c) {
      const bool more = c + 1 < pl.nchunks;
      if (more) {
        if (!prep(c + 1) || !g_and_next_forward(c)) return KD_ERR_CUDA;
      } else if (!g_gemm(c)) {
        return KD_ERR_CUDA;
      }
      if (!dh_and_dw(c)) return KD_ERR_CUDA;
      if (more && !combine(c + 1)) return KD_ERR_CUDA;
    }
    return KD_OK;
  }
  for (int c = 0; c < pl.nchunks; ++c) {
    if (!prep(c)) return KD_ERR_CUDA;
    if (mode & MODE_FWD) {
      if (!forward_gemm(c) || !combine(c)) return KD_ERR_CUDA;
    }
    if (mode & MODE_BWD) {
      if (!keep && !g_gemm(c)) return KD_ERR_CUDA;
      if (!dh_and_dw(c)) return KD_ERR_CUDA;
    }
  }
  return KD_OK;
}

}  // namespace

// ==================================================================== C ABI
extern "C" {

size_t kd_topk_kl_workspace_size(int64_t T, int d, int V, int K, int chunk, int what) {
  Plan pl;
  if (make_plan(T, d, V, K, chunk, what, &pl) != KD_OK) return 0;
  return pl.total;
}

kd_status kd_topk_kl_forward(const void* H, const void* W, const int32_t* idx, const float* p, int64_t T, int d,
                             int V, int K, int chunk, float* loss, float* lse, float* loss_rows, void* workspace,
                             size_t ws_bytes, void* stream) {
  return run(MODE_FWD, H, W, idx, p, nullptr, T, d, V, K, chunk, 1.f, loss, lse, loss_rows, nullptr, nullptr, 0,
             workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

kd_status kd_topk_kl_backward(const void* H, const void* W, const int32_t* idx, const float* p, const float* lse,
                              int64_t T, int d, int V, int K, int chunk, float dloss, float* dH, float* dW,
                              int accumulate_dW, void* workspace, size_t ws_bytes, void* stream) {
  return run(MODE_BWD, H, W, idx, p, lse, T, d, V, K, chunk, dloss, nullptr, nullptr, nullptr, dH, dW,
             accumulate_dW, workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

kd_status kd_topk_kl_fused_step(const void* H, const void* W, const int32_t* idx, const float* p, int64_t T, int d,
                                int V, int K, int chunk, float dloss, float* loss, float* lse, float* loss_rows,
                                float* dH, float* dW, int accumulate_dW, void* workspace, size_t ws_bytes,
                                void* stream) {
  return run(MODE_FWD | MODE_BWD, H, W, idx, p, nullptr, T, d, V, K, chunk, dloss, loss, lse, loss_rows, dH, dW,
             accumulate_dW, workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

kd_status kd_topk_kl_fused_step_norecompute(const void* H, const void* W, const int32_t* idx, const float* p,
                                            int64_t T, int d, int V, int K, int chunk, float dloss, float* loss,
                                            float* lse, float* loss_rows, float* dH, float* dW, int accumulate_dW,
                                            void* workspace, size_t ws_bytes, void* stream) {
  return run(MODE_FWD | MODE_BWD | MODE_KEEP, H, W, idx, p, nullptr, T, d, V, K, chunk, dloss, loss, lse,
             loss_rows, dH, dW, accumulate_dW, workspace, ws_bytes, static_cast<cudaStream_t>(stream));
}

kd_status kd_topk_cache_build(const void* logits, int logits_bf16, int64_t T, int V, int K, int32_t* idx,
                              float* p, float* lse, void* stream) {
  if (!logits || !idx || !p || T < 1 || V < 1 || K < 1 || K > V) return KD_ERR_INVALID_ARG;
  if (K > 1024) return KD_ERR_UNSUPPORTED;
  const uintptr_t need = logits_bf16 ? 1u : 3u;
  if ((reinterpret_cast<uintptr_t>(logits) & need) || (reinterpret_cast<uintptr_t>(idx) & 3u) ||
      (reinterpret_cast<uintptr_t>(p) & 3u) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)))
    return KD_ERR_UNSUPPORTED;
  if (!device_supported()) return KD_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // 16-byte loads when every row starts on a 16-byte boundary
  const bool vec = (reinterpret_cast<uintptr_t>(logits) & 15u) == 0 && (int64_t(V) * (logits_bf16 ? 2 : 4)) % 16 == 0;
  const int sms = current_sm_count();
  const int slot = prof_begin(KD_K_OTHER, st);
  cudaError_t e = cudaSuccess;
  // 32-byte loads when every row is whole 32-byte groups on a 32-byte boundary;
  // the narrow block shape when its slot maxima can bound the K-th key (K <=
  // its slot count) and its group maxima fit (rows of up to 512 KB read 32
  // bytes at a time, 256 KB read 16 bytes at a time)
  const int64_t row_bytes = int64_t(V) * (logits_bf16 ? 2 : 4);
  const bool v32 = vec && (reinterpret_cast<uintptr_t>(logits) & 31u) == 0 && row_bytes % 32 == 0;
  const bool narrow32 = v32 && row_bytes <= 2 * CACHE_WHOLE_ROW && K <= CacheNarrow32::SLOTS;
  const bool narrow = vec && row_bytes <= CACHE_WHOLE_ROW && K <= CacheNarrow::SLOTS;
  // rows whose 16-byte group maxima would not fit the wide shape's shared memory
  const bool wide32 = v32 && row_bytes > int64_t(CacheWide::GMAX) * 16;
  auto run_kernel = [&](auto kern, const auto* z, int threads, int smem) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem) != cudaSuccess || per_sm < 1) {
      cudaGetLastError();
      per_sm = 1;
    }
    const int blocks = static_cast<int>(std::min<int64_t>(T, int64_t(per_sm) * sms));
    kern<<<blocks, threads, smem, st>>>(z, T, V, K, idx, p, lse);
    e = cudaGetLastError();
  };
  auto run_typed = [&](const auto* z) {
    using TL = std::remove_const_t<std::remove_pointer_t<decltype(z)>>;
    if (narrow32)
      run_kernel(kd_topk_cache_kernel<TL, true, CacheNarrow32>, z, CacheNarrow32::NT, CacheNarrow32::smem_bytes(true));
    else if (narrow)
      run_kernel(kd_topk_cache_kernel<TL, true, CacheNarrow>, z, CacheNarrow::NT, CacheNarrow::smem_bytes(true));
    else if (wide32)
      run_kernel(kd_topk_cache_kernel<TL, true, CacheWide32>, z, CacheWide32::NT, CacheWide32::smem_bytes(true));
    else if (vec)
      run_kernel(kd_topk_cache_kernel<TL, true, CacheWide>, z, CacheWide::NT, CacheWide::smem_bytes(true));
    else
      run_kernel(kd_topk_cache_kernel<TL, false, CacheWide>, z, CacheWide::NT, CacheWide::smem_bytes(false));
  };
  if (logits_bf16) run_typed(static_cast<const __nv_bfloat16*>(logits));
  else run_typed(static_cast<const float*>(logits));
  prof_end(slot, st);
  return e == cudaSuccess ? KD_OK : KD_ERR_CUDA;
}

kd_status kd_grad_to_bf16(const float* src, void* dst, int64_t n, float scale, void* stream) {
  if (!src || !dst || n < 0) return KD_ERR_INVALID_ARG;
  if (n == 0) return KD_OK;
  if (!aligned16(src) || (reinterpret_cast<uintptr_t>(dst) & 7u)) return KD_ERR_UNSUPPORTED;
  if (!device_supported()) return KD_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t blocks = std::min<int64_t>(std::max<int64_t>(1, ceil_div(n / 4, 256)), 8L * current_sm_count());
  kd_scale_to_bf16_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(src, static_cast<__nv_bfloat16*>(dst), n,
                                                                         scale);
  return cudaGetLastError() == cudaSuccess ? KD_OK : KD_ERR_CUDA;
}

kd_status kd_topk_kl_device_status(void* workspace, void* stream) {
  if (!workspace) return KD_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int h = 0;
  if (cudaMemcpyAsync(&h, workspace, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return KD_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return KD_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof(int), st) != cudaSuccess) return KD_ERR_CUDA;
  if (h < 0 || h > KD_ERR_CUDA) return KD_ERR_CUDA;
  return static_cast<kd_status>(h);
}

const char* kd_status_string(kd_status s) {
  switch (s) {
    case KD_OK: return "ok";
    case KD_ERR_INVALID_ARG: return "invalid argument";
    case KD_ERR_UNSUPPORTED: return "unsupported shape, alignment or device";
    case KD_ERR_WORKSPACE: return "workspace too small";
    case KD_ERR_BAD_INDEX: return "teacher id outside [0, V)";
    case KD_ERR_TIMEOUT: return "internal pipeline wait timed out";
    case KD_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

kd_status kd_gemm_bf16(const void* A, const void* B, float* D, int M, int N, int K, int lda, int ldb, int ldd,
                       int a_mn, int b_mn, int cta_pair, void* workspace, size_t ws_bytes, void* stream) {
  if (!A || !B || !D || !workspace || M < 1 || N < 1 || K < 1) return KD_ERR_INVALID_ARG;
  if (ws_bytes < 256) return KD_ERR_WORKSPACE;
  if (!aligned16(A) || !aligned16(B) || !aligned16(D) || (lda % 8) || (ldb % 8) || (ldd % 4))
    return KD_ERR_UNSUPPORTED;
  if (lda < (a_mn ? M : K) || ldb < (b_mn ? N : K) || ldd < N) return KD_ERR_INVALID_ARG;
  if (!device_supported()) return KD_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = static_cast<int*>(workspace);
  CUtensorMap ta, tb;
  int a3 = 0, b3 = 0;
  const bool pr = cta_pair != 0;
  bool ok = a_mn ? tmap_bf16_mn(&ta, &a3, A, M, K, uint64_t(lda) * 2, BM)
                 : tmap_bf16(&ta, A, K, M, uint64_t(lda) * 2, BK, BM);
  ok = ok && (b_mn ? tmap_bf16_mn(&tb, &b3, B, N, K, uint64_t(ldb) * 2, pr ? BN / 2 : BN)
                   : tmap_bf16(&tb, B, K, N, uint64_t(ldb) * 2, BK, pr ? BN / 2 : BN));
  CUtensorMap td;
  ok = ok && tmap_f32_out(&td, D, N, M, uint64_t(ldd) * 4);
  if (!ok) return KD_ERR_CUDA;
  if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return KD_ERR_CUDA;
  GemmParams P = base_params(status);
  P.num_m = static_cast<int>(ceil_div(M, pr ? 2 * BM : BM));
  P.num_n = static_cast<int>(ceil_div(N, BN));
  P.kb_total = P.kb_per_split = static_cast<int>(ceil_div(K, BK));
  P.a_mn3d = a3;
  P.b_mn3d = b3;
  const int sms = current_sm_count();
  cudaError_t e;
  if (!a_mn && !b_mn) e = launch_gemm_any<EPI_F32, false, false>(pr, KD_K_OTHER, ta, tb, td, P, sms, st);
  else if (!a_mn && b_mn) e = launch_gemm_any<EPI_F32, false, true>(pr, KD_K_OTHER, ta, tb, td, P, sms, st);
  else if (a_mn && !b_mn) e = launch_gemm_any<EPI_F32, true, false>(pr, KD_K_OTHER, ta, tb, td, P, sms, st);
  else e = launch_gemm_any<EPI_F32, true, true>(pr, KD_K_OTHER, ta, tb, td, P, sms, st);
  return e == cudaSuccess ? KD_OK : KD_ERR_CUDA;
}

kd_status kd_debug_wait_timeout(int wait_limit_ms, int cta_pair, void* workspace, size_t ws_bytes, void* stream) {
  if (!workspace || wait_limit_ms < 1 || wait_limit_ms > 10000) return KD_ERR_INVALID_ARG;
  if (ws_bytes < 256 || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return KD_ERR_WORKSPACE;
  if (!device_supported()) return KD_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* status = static_cast<int*>(workspace);
  // The descriptors are never used to copy anything: the producer withholds every load.
  CUtensorMap ta, tb, td;
  if (!tmap_bf16(&ta, workspace, 64, 1, 128, BK, 1) || !tmap_bf16(&tb, workspace, 64, 1, 128, BK, 1) ||
      !tmap_f32_out(&td, workspace, 32, 1, 128))
    return KD_ERR_CUDA;
  if (cudaMemsetAsync(status, 0, sizeof(int), st) != cudaSuccess) return KD_ERR_CUDA;
  GemmParams P = base_params(status);
  P.wait_limit_ns = static_cast<uint64_t>(wait_limit_ms) * 1000000ull;
  P.debug_withhold_loads = 1;
  P.num_m = 1;
  P.num_n = 1;
  P.kb_total = P.kb_per_split = 2;
  // one CTA, or one pair of CTAs
  if (launch_gemm_any<EPI_F32, false, false>(cta_pair != 0, KD_K_OTHER, ta, tb, td, P, cta_pair ? 2 : 1, st) !=
      cudaSuccess)
    return KD_ERR_CUDA;
  return kd_topk_kl_device_status(workspace, stream);
}

kd_status kd_profile_enable(int on) {
  if (on && g_prof.ev.empty()) {
    g_prof.ev.resize(2 * Profiler::kPairs);
    g_prof.kind.resize(Profiler::kPairs);
    for (auto& e : g_prof.ev)
      if (cudaEventCreate(&e) != cudaSuccess) return KD_ERR_CUDA;
  }
  g_prof.on = on != 0;
  return KD_OK;
}

int kd_profile_read(double* ms_total, int64_t* launches, int n, int reset) {
  double ms[KD_PROF_KINDS] = {0};
  int64_t cnt[KD_PROF_KINDS] = {0};
  for (size_t i = 0; i < g_prof.used; ++i) {
    float t = 0.f;
    if (cudaEventSynchronize(g_prof.ev[2 * i + 1]) == cudaSuccess &&
        cudaEventElapsedTime(&t, g_prof.ev[2 * i], g_prof.ev[2 * i + 1]) == cudaSuccess) {
      ms[g_prof.kind[i]] += t;
      cnt[g_prof.kind[i]] += 1;
    }
  }
  for (int k = 0; k < n && k < KD_PROF_KINDS; ++k) {
    if (ms_total) ms_total[k] = ms[k];
    if (launches) launches[k] = cnt[k];
  }
  if (reset) {
    g_prof.used = 0;
    g_prof.dropped = 0;
  }
  return KD_PROF_KINDS;
}

const char* kd_profile_kind_name(int kind) {
  static const char* names[KD_PROF_KINDS] = {"prep",      "logits_fwd", "combine", "logits_g", "gemm_dh",
                                             "dh_reduce", "gemm_dw",    "other",   "g_from_e", "logits_gf"};
  return (kind >= 0 && kind < KD_PROF_KINDS) ? names[kind] : "unknown";
}

}  // extern "C"

// ==================================================================== forward without allocation
// Some callers cannot call cudaMalloc: a plugin or custom operator that runs
// inside another runtime's device-memory pool and is handed no allocator, a
// process whose device-memory budget is fixed at start-up, or a loop that
// cannot afford the device-wide synchronisation cudaMalloc / cudaFree may
// bring.  For them the forward can run on scratch memory that the library
// itself owns: a file-scope device array, created when the library's device
// code is loaded on a GPU and held by every GPU that loads it until the
// process exits.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB per GPU
__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device; looked up once
// per device (the host-side symbol is only a stand-in, never a device address).
kd_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KD_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return KD_ERR_CUDA;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return KD_OK;
}

}  // namespace

extern "C" kd_status kd_topk_kl_forward_noalloc(const void* H, const void* W, const int32_t* idx, const float* p,
                                                int64_t T, int d, int V, int K, int chunk, float* loss, float* lse,
                                                float* loss_rows, void* stream) {
  Plan pl;
  const kd_status rc = make_plan(T, d, V, K, chunk, KD_WS_FORWARD, &pl);
  if (rc != KD_OK) return rc;
  if (pl.total > kNoAllocScratchBytes) return KD_ERR_WORKSPACE;
  void* scratch = nullptr;
  const kd_status sc = noalloc_scratch(&scratch);
  if (sc != KD_OK) return sc;
  const kd_status lr = kd_topk_kl_forward(H, W, idx, p, T, d, V, K, chunk, loss, lse, loss_rows, scratch,
                                          kNoAllocScratchBytes, stream);
  if (lr != KD_OK) return lr;
  return kd_topk_kl_device_status(scratch, stream);
}
