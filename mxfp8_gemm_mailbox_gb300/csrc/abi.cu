// The C ABI declared in include/mxfp8_mailbox.h: argument checks, the
// publishing-GEMM handle (tensor maps, tactic, launch configuration) and the
// mailbox calls.  Every check happens on the host before a launch; a failed
// check returns a status and leaves a message for mxfp8_last_error().
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "internal.h"
#include "mxfp8_mailbox.h"
#include "noalloc_cache.h"

using namespace mxfp8;

struct mxfp8_publish_gemm {
  mxfp8_gemm_desc desc;  // resolved tactic
  const uint8_t* w;
  uint8_t* w_sf;
  uint8_t* w_tiled;  // nullptr when W is read in place
  uint16_t* mailbox;
  int32_t* state;
  int device;
  // Set by create, whose re-layout kernels write the scale chunks and the
  // tiled weight that the GEMM's producer reads before its grid wait: the
  // first launch then takes a full stream dependency instead of the
  // programmatic one.
  bool first_launch_pending;
  int k_tiles;  // stages of K: ceil(K / (128 fold))
  int tiles_per_split;
  TmemPlan tmem;
  GemmSmemLayout layout;
  CUtensorMap tmap_w;
  // Tensor map of the last activation buffer seen (x pointer, m).
  const void* x_cached;
  int m_cached;
  int32_t x_pieces;  // tmap_x is the 3-D piece view (encode_x)
  CUtensorMap tmap_x;
};

namespace {

thread_local std::string g_last_error;

mxfp8_status fail(mxfp8_status status, const std::string& message) {
  g_last_error = message;
  return status;
}

mxfp8_status cuda_fail(cudaError_t err, const char* what) {
  return fail(MXFP8_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(err));
}

bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

constexpr uint64_t kDefaultPollTimeoutNs = 1000000000ull;
constexpr int kDefaultGemmWaitLimitMs = 2000;
constexpr int kMaxGemmWaitLimitMs = 60000;
// W stages past the ring each CTA warms in L2 by default.  The first 70 % of
// a grid's CTAs launch while the previous kernel streams and warm few; the
// rest warm many.  Measured on GB300, chains of GEMM + consumer rotating
// weights through 14 x the L2: N=7168, K=16384, S=4 (two CTAs per SM) 21.44 us
// per call with 6 stages for every CTA, 20.25 with 4 early and 16 late, best
// among early 0-6, late 8-24 and splits at 36-70 % of the grid; N=7168,
// K=8192, S=2 (one per SM) 13.67 us with 10 for every CTA, 12.98 with none
// early and 16 late.
constexpr int kDefaultL2Prefetch = 16;
constexpr int kDefaultL2PrefetchEarly = 4;          // two CTAs per SM
constexpr int kDefaultL2PrefetchEarlyOnePerSm = -1;  // none
constexpr int kEarlyCtaPercent = 70;
// Tensor-memory columns a CTA may allocate: half of an SM's 512, so two CTAs
// on an SM never wait for each other's allocation.  A third may wait until one
// of them exits: harmless unless they wait for it, which split-K clusters do
// (at their cluster barriers), hence the shared-memory floor of
// at_most_two_per_sm for clustered launches.  A CTA of a later programmatic
// grid never holds columns an earlier one waits for: each CTA allocates before
// it lets its dependents launch.
constexpr uint32_t kMaxTmemCols = 256;

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_tiled() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

// A 2-D uint8 tensor [outer][inner] (row stride `inner` bytes), read in boxes
// of box_outer rows x 128 bytes with the 128-byte swizzle; out-of-range
// elements read as zero.
mxfp8_status encode_rows(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                         uint32_t box_outer) {
  EncodeTiled fn = encode_tiled();
  if (!fn) return fail(MXFP8_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(kTileK), box_outer};
  cuuint32_t elem[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides,
                  box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MXFP8_ERR_CUDA, "cuTensorMapEncodeTiled failed with CUresult " + std::to_string(r));
  return MXFP8_OK;
}

// The activations' tensor map.  Folded tiles (fold > 1) read a stage's fold
// consecutive 128-wide K pieces of the 8 rows; when K is a multiple of 128 a
// 3-D view of x -- (k within a piece, row, piece), strides K and 128 bytes --
// loads them in one box of 128 x 8 x fold, landing piece-major exactly as
// fold boxes of the 2-D view would, so a stage costs one TMA request instead
// of fold.  *pieces tells which view was encoded (the driver may refuse the
// overlapping strides; the 2-D view serves then).
mxfp8_status encode_x(CUtensorMap* map, const void* x, int k, int m, int fold, int32_t* pieces) {
  *pieces = 0;
  if (fold > 1 && k % kTileK == 0) {  // fold here: the pieces of one stage (fold x K tiles)
    EncodeTiled fn = encode_tiled();
    if (!fn) return fail(MXFP8_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kTileK), static_cast<cuuint64_t>(m),
                          static_cast<cuuint64_t>(k / kTileK)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(kTileK)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(kTileK), static_cast<cuuint32_t>(kRows),
                         static_cast<cuuint32_t>(fold)};
    cuuint32_t elem[3] = {1, 1, 1};
    if (fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(x), dims, strides, box, elem,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS) {
      *pieces = 1;
      return MXFP8_OK;
    }
  }
  return encode_rows(map, x, static_cast<uint64_t>(k), static_cast<uint64_t>(m), kRows);
}

mxfp8_status check_desc(const mxfp8_gemm_desc* d) {
  if (!d) return fail(MXFP8_ERR_INVALID, "desc is NULL");
  if (d->n <= 0 || d->n % kBlockN)
    return fail(MXFP8_ERR_INVALID, "n must be a positive multiple of 128, got " + std::to_string(d->n));
  if (d->k <= 0 || d->k % 32)
    return fail(MXFP8_ERR_INVALID, "k must be a positive multiple of 32, got " + std::to_string(d->k));
  if (d->k > 32768) return fail(MXFP8_ERR_UNSUPPORTED, "k above 32768 is not supported");
  if (d->capacity_m < 1 || d->capacity_m > MXFP8_MAX_ROWS)
    return fail(MXFP8_ERR_INVALID, "capacity_m must be in 1..8");
  if (d->split_k != 0 && d->split_k != 1 && d->split_k != 2 && d->split_k != 4 &&
      d->split_k != 8)
    return fail(MXFP8_ERR_UNSUPPORTED, "split_k must be 1, 2, 4 or 8 (or 0 to choose)");
  if (d->cta_k != 0 && d->cta_k != kTileK && d->cta_k != 2 * kTileK)
    return fail(MXFP8_ERR_UNSUPPORTED, "cta_k must be 128 or 256 (or 0 for 128)");
  if (d->cta_k == 2 * kTileK) {
    if (d->fold == 8) return fail(MXFP8_ERR_UNSUPPORTED, "cta_k 256 takes fold 1, 2 or 4");
    if (d->split_k == 8) return fail(MXFP8_ERR_UNSUPPORTED, "cta_k 256 takes split_k 1, 2 or 4");
    if (d->acc_blocks == 1)
      return fail(MXFP8_ERR_UNSUPPORTED, "cta_k 256 takes acc_blocks 4 (one slot per K tile)");
    if (d->tmem_load == MXFP8_TMEM_LOAD_16X256B)
      return fail(MXFP8_ERR_UNSUPPORTED, "cta_k 256 reads accumulators with 32x32b");
  }
  if (d->stages != 0 && (d->stages < 2 || d->stages > kMaxStages))
    return fail(MXFP8_ERR_UNSUPPORTED, "stages must be in 2..16 (or 0 to choose)");
  if (d->acc_blocks != 0 && d->acc_blocks != 1 && d->acc_blocks != 4)
    return fail(MXFP8_ERR_UNSUPPORTED, "acc_blocks must be 1 or 4 (or 0 to choose)");
  if (d->w_layout != 0 && d->w_layout != MXFP8_W_IN_PLACE && d->w_layout != MXFP8_W_TILED)
    return fail(MXFP8_ERR_UNSUPPORTED, "w_layout must be MXFP8_W_IN_PLACE or MXFP8_W_TILED");
  if (d->l2_prefetch < -1 || d->l2_prefetch > 64)
    return fail(MXFP8_ERR_UNSUPPORTED, "l2_prefetch must be in 1..64, -1 (none) or 0 (choose)");
  if (d->l2_prefetch_early < -1 || d->l2_prefetch_early > 64)
    return fail(MXFP8_ERR_UNSUPPORTED,
                "l2_prefetch_early must be in 1..64, -1 (none) or 0 (choose)");
  if (d->pipes != 0 && d->pipes != 1 && d->pipes != 2 && d->pipes != 4)
    return fail(MXFP8_ERR_UNSUPPORTED, "pipes must be 1, 2 or 4 (or 0 to choose)");
  if (d->tmem_load != 0 && d->tmem_load != MXFP8_TMEM_LOAD_32X32B &&
      d->tmem_load != MXFP8_TMEM_LOAD_16X256B)
    return fail(MXFP8_ERR_UNSUPPORTED,
                "tmem_load must be MXFP8_TMEM_LOAD_32X32B or MXFP8_TMEM_LOAD_16X256B");
  if (d->fold != 0 && d->fold != 1 && d->fold != 2 && d->fold != 4 && d->fold != 8)
    return fail(MXFP8_ERR_UNSUPPORTED, "fold must be 1, 2, 4 or 8 (or 0 to choose)");
  if (d->wait_limit_ms < 0 || d->wait_limit_ms > kMaxGemmWaitLimitMs)
    return fail(MXFP8_ERR_UNSUPPORTED, "wait_limit_ms must be in 1.." +
                                           std::to_string(kMaxGemmWaitLimitMs) + " (or 0 for " +
                                           std::to_string(kDefaultGemmWaitLimitMs) + ")");
  if (d->fold == 8) {
    if (d->split_k > 1) return fail(MXFP8_ERR_UNSUPPORTED, "fold 8 takes split_k 1");
    if (d->pipes == 4)
      return fail(MXFP8_ERR_UNSUPPORTED,
                  "fold 8 takes at most 2 pipes (its accumulator ring has 2 slots)");
  }
  if (d->fold > 1) {
    if (d->split_k == 8)
      return fail(MXFP8_ERR_UNSUPPORTED, "fold > 1 takes split_k 1, 2 or 4");
    if (d->acc_blocks == 1)
      return fail(MXFP8_ERR_UNSUPPORTED,
                  "fold > 1 takes acc_blocks 4 (one slot per MMA does not fit in tensor memory)");
    if (d->tmem_load == MXFP8_TMEM_LOAD_16X256B)
      return fail(MXFP8_ERR_UNSUPPORTED, "fold > 1 reads accumulators with 32x32b");
  }
  return MXFP8_OK;
}

// The fold a descriptor's buffers are sized for: 0 (choose) picks only folds
// that pad K no further than 1 does, so it sizes like 1.
int sizing_fold(int fold) { return fold == 0 ? 1 : fold; }

int resolved_w_layout(int w_layout) { return w_layout == 0 ? MXFP8_W_TILED : w_layout; }

size_t scale_chunk_bytes(int n, int k, int fold) {
  return static_cast<size_t>(n / (kBlockN / fold)) * k_tiles_for_fold(k, fold) * kSfChunkBytes;
}

size_t tiled_w_offset(int n, int k, int fold) {
  return (scale_chunk_bytes(n, k, fold) + 255) & ~size_t{255};
}

struct DeviceLimits {
  int sms = 0;
  int smem_optin = 0;
  int smem_per_sm = 0;
};

mxfp8_status device_limits(int device, DeviceLimits* out) {
  cudaError_t e;
  if ((e = cudaDeviceGetAttribute(&out->sms, cudaDevAttrMultiProcessorCount, device)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
  if ((e = cudaDeviceGetAttribute(&out->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                  device)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute(shared memory per block)");
  if ((e = cudaDeviceGetAttribute(&out->smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                  device)) != cudaSuccess)
    return cuda_fail(e, "cudaDeviceGetAttribute(shared memory per SM)");
  return MXFP8_OK;
}

// A clustered launch (split_k > 1) asks for at least a third of an SM's shared
// memory, so at most two of its CTAs share an SM and none waits in tcgen05.alloc
// for columns held by a cluster peer that waits for it.  (Unclustered short
// rings stay small: the padding costs latency-bound shapes about 0.35 us.)
GemmSmemLayout at_most_two_per_sm(GemmSmemLayout layout, int split_k, const DeviceLimits& lim) {
  if (split_k > 1)
    layout.total = std::max(layout.total, static_cast<uint32_t>(lim.smem_per_sm / 3));
  return layout;
}

// The dynamic shared-memory limit of a kernel instantiation is one value per
// device, shared by every handle (and allocation-free call) that launches it.
// It only bounds what a launch may ask for, so it is raised to the largest
// size any of them needs and never lowered: a handle with a shallower ring
// must not push it below an earlier handle's launch size.  `force` sets it
// again even when the recorded value suffices (precompile does, so a context
// that was torn down and re-created gets it back).
constexpr int kMaxDevicesTracked = 64;

mxfp8_status ensure_smem_attribute(int device, int split_k, int fold, int tiles_per_stage,
                                   int bytes, bool force) {
  static std::mutex mutex;
  // [device][log2 split_k][log2 fold][tiles per stage - 1]: split_k and fold
  // are 1, 2, 4 or 8, tiles per stage 1 or 2.
  static int raised[kMaxDevicesTracked][4][4][2] = {};
  if (device < 0 || device >= kMaxDevicesTracked)
    return fail(MXFP8_ERR_UNSUPPORTED, "device ordinal out of range for the launch table");
  const int si = split_k == 8 ? 3 : split_k / 2;
  const int fi = fold == 8 ? 3 : fold / 2;
  std::lock_guard<std::mutex> lock(mutex);
  int& have = raised[device][si][fi][tiles_per_stage == 2 ? 1 : 0];
  if (!force && have >= bytes) return MXFP8_OK;
  const int want = std::max(have, bytes);
  const cudaError_t e = set_gemm_smem_attribute(split_k, fold, want, tiles_per_stage);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(max dynamic shared memory)");
  have = want;
  return MXFP8_OK;
}

// The launch's shared-memory layout for a resolved descriptor.  With split-K
// the partials from peers get a region of their own when it fits beside the
// resolved ring (within the same per-SM budget the ring was sized for): a CTA
// then sends its partials as soon as its main loop is done instead of waiting
// at a cluster barrier until every peer's ring is dead.
GemmSmemLayout launch_layout(const mxfp8_gemm_desc& d, int tiles_per_split,
                             const DeviceLimits& lim) {
  const int T = d.cta_k / kTileK;
  GemmSmemLayout layout = gemm_smem_layout(d.stages, d.split_k, tiles_per_split, d.fold, false, T);
  if (d.split_k > 1) {
    const int ctas = d.n / (kBlockN / d.fold) * d.split_k;
    const int budget = ctas > lim.sms ? lim.smem_per_sm / 2 - 1024 : lim.smem_optin;
    const GemmSmemLayout own =
        gemm_smem_layout(d.stages, d.split_k, tiles_per_split, d.fold, true, T);
    if (static_cast<int>(own.total) <= budget) layout = own;
  }
  return at_most_two_per_sm(layout, d.split_k, lim);
}

// Fill split_k, cta_k, stages, pipes and fold: split_k so the grid has about
// one or two CTAs per SM; then the largest fold that keeps at most one CTA
// per SM (one SM streams only so fast: few-CTA grids leave HBM idle); the
// deepest ring that still lets the intended number of CTAs share an SM,
// rounded so the pipes divide it: with at most one CTA per SM each CTA must
// stream fast, so 4 pipes (ring a multiple of 4); with two, HBM is the limit
// and 2 pipes suffice (more in flight measured slower).
mxfp8_status resolve_tactic(mxfp8_gemm_desc* d, const DeviceLimits& lim) {
  const int tiles = d->n / kBlockN;
  const int k_tiles1 = k_tiles_for_fold(d->k, 1);
  if (d->split_k == 0) {
    int s = 1;
    for (int cand : {2, 4})  // 8 measured slower than 4 on every shape where both fit
      if (tiles * cand <= 2 * lim.sms && k_tiles1 >= 2 * cand) s = cand;
    d->split_k = s;
  }
  if (d->cta_k == 0) d->cta_k = kTileK;
  const int T = d->cta_k / kTileK;  // K tiles per pipeline stage
  if (d->wait_limit_ms == 0) d->wait_limit_ms = kDefaultGemmWaitLimitMs;
  if (d->acc_blocks == 0) d->acc_blocks = 4;
  if (d->tmem_load == 0) d->tmem_load = MXFP8_TMEM_LOAD_32X32B;
  d->w_layout = resolved_w_layout(d->w_layout);
  if (d->fold == 0) {
    int f = 1;
    const bool foldable = d->split_k <= 4 && d->acc_blocks == 4 &&
                          d->tmem_load == MXFP8_TMEM_LOAD_32X32B;
    for (int cand : {2, 4, 8}) {
      // Fold 8 (unsplit, two pipes at most) pays from 8 stages per CTA on
      // (measured on GB300, N=2048, S=1: K=4096 6.29 vs 6.00 us at fold 4,
      // K=8192 7.86 vs 8.79, K=16384 11.46 vs 13.60).
      if (cand == 8 &&
          (d->split_k != 1 || d->pipes == 4 || k_tiles_for_fold(d->k, 8) < 8 || T != 1))
        continue;
      if (foldable && tiles * d->split_k * cand <= lim.sms &&
          k_tiles_for_fold(d->k, cand) * cand == k_tiles1 &&  // no more K padding
          k_tiles_for_fold(d->k, cand) >= d->split_k)          // a full stage per split
        f = cand;
    }
    d->fold = f;
  }
  if (d->fold == 8 && d->split_k != 1) return fail(MXFP8_ERR_UNSUPPORTED, "fold 8 takes split_k 1");
  const int k_tiles = k_tiles_for_fold(d->k, d->fold);
  const int tps = (k_tiles + d->split_k - 1) / d->split_k;
  if (tps * d->fold > kMaxTilesPerSplit)
    return fail(MXFP8_ERR_UNSUPPORTED, "too many K tiles per split: raise split_k");
  const int ctas = tiles * d->fold * d->split_k;
  const int per_sm = ctas > lim.sms ? 2 : 1;
  const int budget = per_sm == 2 ? lim.smem_per_sm / 2 - 1024 : lim.smem_optin;
  if (d->l2_prefetch_early == 0)
    d->l2_prefetch_early = d->l2_prefetch != 0 ? d->l2_prefetch
                           : per_sm == 2       ? kDefaultL2PrefetchEarly
                                               : kDefaultL2PrefetchEarlyOnePerSm;
  if (d->l2_prefetch == 0) d->l2_prefetch = kDefaultL2Prefetch;
  if (d->stages == 0) {
    int best = 0;
    for (int s = 2; s <= kMaxStages; ++s) {
      if (static_cast<int>(gemm_smem_layout(s, d->split_k, tps, d->fold, false, T).total) >
          budget)
        break;
      if (gemm_tmem_plan(s, d->acc_blocks, d->fold, T).cols > kMaxTmemCols) break;
      best = s;
      if (s * T >= tps) break;  // more stages than K tiles buy nothing
    }
    if (best == 0) return fail(MXFP8_ERR_UNSUPPORTED, "no stage count fits in shared memory");
    const int unit = (per_sm == 1 && best >= 4) ? 4 : (best >= 2 ? 2 : 1);
    best -= best % unit;
    d->stages = best;
  }
  if (static_cast<int>(gemm_smem_layout(d->stages, d->split_k, tps, d->fold, false, T).total) >
      lim.smem_optin)
    return fail(MXFP8_ERR_UNSUPPORTED, "the requested stages do not fit in shared memory");
  const TmemPlan tmem = gemm_tmem_plan(d->stages, d->acc_blocks, d->fold, T);
  if (tmem.cols > kMaxTmemCols)
    return fail(MXFP8_ERR_UNSUPPORTED, "the requested stages do not fit in tensor memory");
  // Every accumulator slot keeps one issuer: the ring (of K tiles) is a
  // multiple of the K tiles the issuers take per round, T pipes.
  const int acc_ring = static_cast<int>(tmem.acc_ring);
  if (d->pipes == 0) {
    d->pipes = (per_sm == 1 && d->stages % 4 == 0 && d->fold != 8) ? 4
               : (d->stages % 2 == 0 ? 2 : 1);
    while (d->pipes > 1 && acc_ring % (T * d->pipes) != 0) d->pipes /= 2;
  } else if (d->stages % d->pipes != 0) {
    return fail(MXFP8_ERR_UNSUPPORTED, "pipes must divide stages (stage i and its ring slots "
                                       "belong to pipe i % pipes)");
  } else if (acc_ring % (T * d->pipes) != 0) {
    return fail(MXFP8_ERR_UNSUPPORTED,
                "with cta_k 256 the accumulator ring (" + std::to_string(acc_ring) +
                    " slots) must be a multiple of 2 x pipes");
  }
  return MXFP8_OK;
}

// The grid's first CTAs, which launch while the previous kernel still runs.
int32_t early_ctas_of(const mxfp8_gemm_desc& d) {
  const int ctas = d.n / (kBlockN / d.fold) * d.split_k;
  return static_cast<int32_t>(ctas * kEarlyCtaPercent / 100);
}

mxfp8_status check_rows(const mxfp8_publish_gemm* g, int32_t m) {
  const int limit = std::min(MXFP8_MAX_ROWS, static_cast<int>(g->desc.capacity_m));
  if (m < 1 || m > limit)
    return fail(MXFP8_ERR_UNSUPPORTED,
                "m must be in 1.." + std::to_string(limit) + ", got " + std::to_string(m));
  return MXFP8_OK;
}

mxfp8_status run_gemm(mxfp8_publish_gemm* g, const void* x, const void* x_scale, int32_t m,
                      void* c, void* stream, bool publish, const float* alpha = nullptr) {
  if (!g) return fail(MXFP8_ERR_INVALID, "gemm handle is NULL");
  mxfp8_status st = check_rows(g, m);
  if (st != MXFP8_OK) return st;
  if (!x || !aligned(x, 16)) return fail(MXFP8_ERR_INVALID, "x must be a 16-byte aligned device pointer");
  if (!x_scale) return fail(MXFP8_ERR_INVALID, "x_scale is NULL");
  if (c && !aligned(c, 16)) return fail(MXFP8_ERR_INVALID, "c must be 16-byte aligned");
  if (!publish && !c) return fail(MXFP8_ERR_INVALID, "the unfused GEMM needs c");
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess || device != g->device)
    return fail(MXFP8_ERR_INVALID, "the handle was created on device " + std::to_string(g->device) +
                                       ", the current device is " + std::to_string(device));
  if (g->x_cached != x || g->m_cached != m) {
    st = encode_x(&g->tmap_x, x, g->desc.k, m, g->desc.fold * (g->desc.cta_k / kTileK),
                  &g->x_pieces);
    if (st != MXFP8_OK) return st;
    g->x_cached = x;
    g->m_cached = m;
  }
  GemmParams p{};
  p.n = g->desc.n;
  p.k = g->desc.k;
  p.m = m;
  p.k_tiles = g->k_tiles;
  p.tiles_per_split = g->tiles_per_split;
  p.stages = g->desc.stages;
  p.capacity = g->desc.capacity_m;
  p.publish = publish ? 1 : 0;
  p.acc_blocks = g->desc.acc_blocks;
  p.l2_prefetch = std::max(0, static_cast<int>(g->desc.l2_prefetch));
  p.l2_prefetch_early = std::max(0, static_cast<int>(g->desc.l2_prefetch_early));
  p.early_ctas = early_ctas_of(g->desc);
  p.pipes = g->desc.pipes;
  p.tmem_load = g->desc.tmem_load;
  p.fold = g->desc.fold;
  p.x_pieces = g->x_pieces;
  p.tiles_per_stage = g->desc.cta_k / kTileK;
  p.tmem = g->tmem;
  p.x_scale = static_cast<const uint8_t*>(x_scale);
  p.w_sf = g->w_sf;
  p.w_tiled = g->w_tiled;
  p.c = static_cast<uint16_t*>(c);
  p.alpha = alpha;
  p.mailbox = g->mailbox;
  p.state = g->state;
  p.wait_limit_ns = static_cast<uint64_t>(g->desc.wait_limit_ms) * 1000000ull;
  p.smem = g->layout;
  cudaError_t e = launch_publish_gemm(g->tmap_w, g->tmap_x, p, g->desc.split_k,
                                      static_cast<cudaStream_t>(stream),
                                      !g->first_launch_pending);
  if (e != cudaSuccess) return cuda_fail(e, "launching the publishing GEMM");
  g->first_launch_pending = false;
  return MXFP8_OK;
}

mxfp8_status check_mailbox(const void* mailbox, const int32_t* state, int32_t capacity_m,
                           int32_t n) {
  if (!mailbox || !aligned(mailbox, 16))
    return fail(MXFP8_ERR_INVALID, "mailbox must be a 16-byte aligned device pointer");
  if (!state || !aligned(state, 16))
    return fail(MXFP8_ERR_INVALID, "stage_state must be a 16-byte aligned device int32[4]");
  if (capacity_m < 1 || capacity_m > MXFP8_MAX_ROWS)
    return fail(MXFP8_ERR_INVALID, "capacity_m must be in 1..8");
  if (n <= 0 || n % 8) return fail(MXFP8_ERR_INVALID, "n must be a positive multiple of 8");
  return MXFP8_OK;
}

}  // namespace

extern "C" {

size_t mxfp8_mailbox_bytes(int32_t capacity_m, int32_t n) {
  if (capacity_m < 1 || capacity_m > MXFP8_MAX_ROWS || n <= 0 || n % 8) return 0;
  return static_cast<size_t>(MXFP8_MAILBOX_GENERATIONS) * capacity_m * n * 2;
}

mxfp8_status mxfp8_mailbox_init(void* mailbox, int32_t* stage_state, int32_t capacity_m,
                                int32_t n, void* stream) {
  mxfp8_status st = check_mailbox(mailbox, stage_state, capacity_m, n);
  if (st != MXFP8_OK) return st;
  cudaError_t e = launch_mailbox_init(static_cast<uint16_t*>(mailbox), stage_state, capacity_m, n,
                                      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "launching the mailbox init kernel");
  return MXFP8_OK;
}

size_t mxfp8_publish_gemm_workspace_bytes(const mxfp8_gemm_desc* desc) {
  if (!desc || desc->n <= 0 || desc->n % kBlockN || desc->k <= 0 || desc->k % 32) return 0;
  if (desc->fold != 0 && desc->fold != 1 && desc->fold != 2 && desc->fold != 4 &&
      desc->fold != 8)
    return 0;
  const int fold = sizing_fold(desc->fold);
  if (resolved_w_layout(desc->w_layout) != MXFP8_W_TILED)
    return scale_chunk_bytes(desc->n, desc->k, fold);
  return tiled_w_offset(desc->n, desc->k, fold) +
         static_cast<size_t>(desc->n / (kBlockN / fold)) * k_tiles_for_fold(desc->k, fold) *
             kWTileBytes;
}

mxfp8_status mxfp8_publish_gemm_create(const mxfp8_gemm_desc* desc, const void* w,
                                       const void* w_scale, void* mailbox,
                                       int32_t* stage_state, void* workspace,
                                       size_t workspace_bytes, void* stream,
                                       mxfp8_publish_gemm** out) {
  if (!out) return fail(MXFP8_ERR_INVALID, "out is NULL");
  *out = nullptr;
  mxfp8_status st = check_desc(desc);
  if (st != MXFP8_OK) return st;
  if (!w || !aligned(w, 16)) return fail(MXFP8_ERR_INVALID, "w must be a 16-byte aligned device pointer");
  if (!w_scale) return fail(MXFP8_ERR_INVALID, "w_scale is NULL");
  st = check_mailbox(mailbox, stage_state, desc->capacity_m, desc->n);
  if (st != MXFP8_OK) return st;
  const size_t need = mxfp8_publish_gemm_workspace_bytes(desc);
  if (!workspace || !aligned(workspace, 16))
    return fail(MXFP8_ERR_INVALID, "workspace must be a 16-byte aligned device pointer");
  if (workspace_bytes < need)
    return fail(MXFP8_ERR_INVALID, "workspace too small: need " + std::to_string(need) + " bytes");

  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  DeviceLimits lim;
  st = device_limits(device, &lim);
  if (st != MXFP8_OK) return st;

  mxfp8_publish_gemm* g = new (std::nothrow) mxfp8_publish_gemm();
  if (!g) return fail(MXFP8_ERR_INVALID, "out of host memory");
  g->desc = *desc;
  st = resolve_tactic(&g->desc, lim);
  if (st != MXFP8_OK) {
    delete g;
    return st;
  }
  g->w = static_cast<const uint8_t*>(w);
  g->w_sf = static_cast<uint8_t*>(workspace);
  const int fold = g->desc.fold;
  g->w_tiled = g->desc.w_layout == MXFP8_W_TILED
                   ? static_cast<uint8_t*>(workspace) + tiled_w_offset(desc->n, desc->k, fold)
                   : nullptr;
  g->mailbox = static_cast<uint16_t*>(mailbox);
  g->state = stage_state;
  g->device = device;
  g->first_launch_pending = true;
  g->k_tiles = k_tiles_for_fold(desc->k, fold);
  g->tiles_per_split = (g->k_tiles + g->desc.split_k - 1) / g->desc.split_k;
  g->tmem = gemm_tmem_plan(g->desc.stages, g->desc.acc_blocks, fold, g->desc.cta_k / kTileK);
  g->layout = launch_layout(g->desc, g->tiles_per_split, lim);
  g->x_cached = nullptr;
  g->m_cached = 0;
  st = encode_rows(&g->tmap_w, w, static_cast<uint64_t>(desc->k), static_cast<uint64_t>(desc->n),
                   kBlockN / fold);
  if (st != MXFP8_OK) {
    delete g;
    return st;
  }
  st = ensure_smem_attribute(device, g->desc.split_k, fold, g->desc.cta_k / kTileK,
                             static_cast<int>(g->layout.total), false);
  if (st != MXFP8_OK) {
    delete g;
    return st;
  }
  e = launch_relayout_w_scales(static_cast<const uint8_t*>(w_scale), g->w_sf, desc->n, desc->k,
                               fold, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    delete g;
    return cuda_fail(e, "launching the W scale re-layout");
  }
  if (g->w_tiled != nullptr) {
    e = launch_tile_weights(static_cast<const uint8_t*>(w), g->w_tiled, desc->n, desc->k, fold,
                            static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
      delete g;
      return cuda_fail(e, "launching the W tiling copy");
    }
  }
  *out = g;
  return MXFP8_OK;
}

mxfp8_status mxfp8_publish_gemm_config(const mxfp8_publish_gemm* gemm, mxfp8_gemm_desc* desc,
                                       int32_t* smem_bytes, int32_t* tmem_columns,
                                       int32_t* grid_ctas) {
  if (!gemm) return fail(MXFP8_ERR_INVALID, "gemm handle is NULL");
  if (desc) *desc = gemm->desc;
  if (smem_bytes) *smem_bytes = static_cast<int32_t>(gemm->layout.total);
  if (tmem_columns) *tmem_columns = static_cast<int32_t>(gemm->tmem.cols);
  if (grid_ctas)
    *grid_ctas = (gemm->desc.n / (kBlockN / gemm->desc.fold)) * gemm->desc.split_k;
  return MXFP8_OK;
}

mxfp8_status mxfp8_publish_gemm_plan(const mxfp8_gemm_desc* desc, int32_t sms,
                                     int32_t smem_per_sm, int32_t smem_per_block_optin,
                                     mxfp8_gemm_desc* resolved, int32_t* smem_bytes,
                                     int32_t* tmem_columns, int32_t* grid_ctas) {
  mxfp8_status st = check_desc(desc);
  if (st != MXFP8_OK) return st;
  if (sms <= 0 || smem_per_sm <= 0 || smem_per_block_optin <= 0)
    return fail(MXFP8_ERR_INVALID, "device limits must be positive");
  DeviceLimits lim;
  lim.sms = sms;
  lim.smem_per_sm = smem_per_sm;
  lim.smem_optin = smem_per_block_optin;
  mxfp8_gemm_desc d = *desc;
  st = resolve_tactic(&d, lim);
  if (st != MXFP8_OK) return st;
  const int k_tiles = k_tiles_for_fold(d.k, d.fold);
  const int tiles_per_split = (k_tiles + d.split_k - 1) / d.split_k;
  const GemmSmemLayout layout = launch_layout(d, tiles_per_split, lim);
  if (resolved) *resolved = d;
  if (smem_bytes) *smem_bytes = static_cast<int32_t>(layout.total);
  if (tmem_columns)
    *tmem_columns =
        static_cast<int32_t>(gemm_tmem_plan(d.stages, d.acc_blocks, d.fold, d.cta_k / kTileK).cols);
  if (grid_ctas) *grid_ctas = (d.n / (kBlockN / d.fold)) * d.split_k;
  return MXFP8_OK;
}

mxfp8_status mxfp8_publish_gemm_precompile(mxfp8_publish_gemm* gemm, int32_t m) {
  if (!gemm) return fail(MXFP8_ERR_INVALID, "gemm handle is NULL");
  mxfp8_status st = check_rows(gemm, m);
  if (st != MXFP8_OK) return st;
  if (!encode_tiled()) return fail(MXFP8_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  return ensure_smem_attribute(gemm->device, gemm->desc.split_k, gemm->desc.fold,
                               gemm->desc.cta_k / kTileK, static_cast<int>(gemm->layout.total),
                               true);
}

mxfp8_status mxfp8_publish_gemm_run(mxfp8_publish_gemm* gemm, const void* x, const void* x_scale,
                                    int32_t m, void* c, void* stream) {
  return run_gemm(gemm, x, x_scale, m, c, stream, true);
}

mxfp8_status mxfp8_publish_gemm_run_scaled(mxfp8_publish_gemm* gemm, const void* x,
                                           const void* x_scale, int32_t m, const float* alpha,
                                           void* c, void* stream) {
  if (alpha && !aligned(alpha, 4)) return fail(MXFP8_ERR_INVALID, "alpha must be 4-byte aligned");
  return run_gemm(gemm, x, x_scale, m, c, stream, true, alpha);
}

mxfp8_status mxfp8_gemm_run_unfused(mxfp8_publish_gemm* gemm, const void* x, const void* x_scale,
                                    int32_t m, void* c, void* stream) {
  return run_gemm(gemm, x, x_scale, m, c, stream, false);
}

mxfp8_status mailbox_publish(void* mailbox, int32_t* stage_state, int32_t capacity_m, int32_t n,
                             int32_t m, const void* c, void* stream) {
  mxfp8_status st = check_mailbox(mailbox, stage_state, capacity_m, n);
  if (st != MXFP8_OK) return st;
  if (m < 1 || m > capacity_m) return fail(MXFP8_ERR_UNSUPPORTED, "m must be in 1..capacity_m");
  if (!c || !aligned(c, 16)) return fail(MXFP8_ERR_INVALID, "c must be a 16-byte aligned device pointer");
  cudaError_t e = launch_mailbox_publish(static_cast<uint16_t*>(mailbox), stage_state, capacity_m,
                                         n, m, static_cast<const uint16_t*>(c),
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "launching the publish kernel");
  return MXFP8_OK;
}

mxfp8_status mailbox_consume(void* mailbox, int32_t* stage_state, int32_t capacity_m, int32_t n,
                             int32_t m, void* out, uint64_t timeout_ns, void* stream) {
  mxfp8_status st = check_mailbox(mailbox, stage_state, capacity_m, n);
  if (st != MXFP8_OK) return st;
  if (m < 1 || m > capacity_m) return fail(MXFP8_ERR_UNSUPPORTED, "m must be in 1..capacity_m");
  if (!out || !aligned(out, 16)) return fail(MXFP8_ERR_INVALID, "out must be a 16-byte aligned device pointer");
  cudaError_t e = launch_mailbox_consume(static_cast<uint16_t*>(mailbox), stage_state, capacity_m,
                                         n, m, static_cast<uint16_t*>(out),
                                         timeout_ns ? timeout_ns : kDefaultPollTimeoutNs,
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "launching the consumer");
  return MXFP8_OK;
}

size_t tagged_mailbox_bytes(int32_t capacity_m, int32_t n) {
  if (capacity_m < 1 || capacity_m > MXFP8_MAX_ROWS || n <= 0 || n % 8) return 0;
  return static_cast<size_t>(capacity_m) * n * 4;
}

mxfp8_status tagged_mailbox_init(void* pairs, int32_t capacity_m, int32_t n, void* stream) {
  const size_t bytes = tagged_mailbox_bytes(capacity_m, n);
  if (bytes == 0) return fail(MXFP8_ERR_INVALID, "capacity_m must be in 1..8 and n a multiple of 8");
  if (!pairs || !aligned(pairs, 16))
    return fail(MXFP8_ERR_INVALID, "pairs must be a 16-byte aligned device pointer");
  cudaError_t e = launch_tagged_init(pairs, bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "launching the tagged mailbox init");
  return MXFP8_OK;
}

mxfp8_status tagged_publish(void* pairs, int32_t capacity_m, int32_t n, int32_t m, const void* c,
                            uint32_t tag, void* stream) {
  if (tagged_mailbox_bytes(capacity_m, n) == 0)
    return fail(MXFP8_ERR_INVALID, "capacity_m must be in 1..8 and n a multiple of 8");
  if (m < 1 || m > capacity_m) return fail(MXFP8_ERR_UNSUPPORTED, "m must be in 1..capacity_m");
  if (tag == 0) return fail(MXFP8_ERR_INVALID, "tag 0 is the armed state; use a nonzero epoch");
  if (!pairs || !aligned(pairs, 16) || !c || !aligned(c, 16))
    return fail(MXFP8_ERR_INVALID, "pairs and c must be 16-byte aligned device pointers");
  cudaError_t e = launch_tagged_publish(pairs, n, m, static_cast<const uint16_t*>(c), tag,
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "launching the tagged publish");
  return MXFP8_OK;
}

mxfp8_status tagged_consume(void* pairs, int32_t capacity_m, int32_t n, int32_t m, uint32_t tag,
                            void* out, uint64_t timeout_ns, int32_t* flags, void* stream) {
  if (tagged_mailbox_bytes(capacity_m, n) == 0)
    return fail(MXFP8_ERR_INVALID, "capacity_m must be in 1..8 and n a multiple of 8");
  if (m < 1 || m > capacity_m) return fail(MXFP8_ERR_UNSUPPORTED, "m must be in 1..capacity_m");
  if (tag == 0) return fail(MXFP8_ERR_INVALID, "tag 0 is the armed state; use a nonzero epoch");
  if (!pairs || !aligned(pairs, 16) || !out || !aligned(out, 16))
    return fail(MXFP8_ERR_INVALID, "pairs and out must be 16-byte aligned device pointers");
  if (flags && !aligned(flags, 4)) return fail(MXFP8_ERR_INVALID, "flags must be 4-byte aligned");
  cudaError_t e = launch_tagged_consume(pairs, n, m, tag, static_cast<uint16_t*>(out),
                                        timeout_ns ? timeout_ns : kDefaultPollTimeoutNs, flags,
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "launching the tagged consume");
  return MXFP8_OK;
}

size_t lamport_gather_mailbox_bytes(size_t capacity_bytes) {
  if (capacity_bytes == 0 || capacity_bytes % 16 || capacity_bytes > MXFP8_GATHER_MAX_CAPACITY)
    return 0;
  return static_cast<size_t>(MXFP8_MAILBOX_GENERATIONS) * capacity_bytes;
}

mxfp8_status lamport_gather_init(void* mailbox, int32_t* state, size_t capacity_bytes,
                                 void* stream) {
  if (lamport_gather_mailbox_bytes(capacity_bytes) == 0)
    return fail(MXFP8_ERR_INVALID, "the capacity must be a positive multiple of 16 bytes, at most " +
                                       std::to_string(MXFP8_GATHER_MAX_CAPACITY));
  if (!mailbox || !aligned(mailbox, 16))
    return fail(MXFP8_ERR_INVALID, "mailbox must be a 16-byte aligned device pointer");
  if (!state || !aligned(state, 16))
    return fail(MXFP8_ERR_INVALID, "state must be a 16-byte aligned device int32[4]");
  cudaError_t e = launch_lamport_gather_init(mailbox, state, capacity_bytes,
                                             static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "launching the gather mailbox init");
  return MXFP8_OK;
}

mxfp8_status lamport_all_gather(void* mailbox, int32_t* state, size_t capacity_bytes,
                                const void* in, size_t nbytes, void* out, uint64_t timeout_ns,
                                void* stream) {
  if (lamport_gather_mailbox_bytes(capacity_bytes) == 0)
    return fail(MXFP8_ERR_INVALID, "the capacity must be a positive multiple of 16 bytes, at most " +
                                       std::to_string(MXFP8_GATHER_MAX_CAPACITY));
  if (nbytes == 0 || nbytes % 16 || nbytes > capacity_bytes)
    return fail(MXFP8_ERR_INVALID, "the gather takes 16-byte multiples of up to " +
                                       std::to_string(capacity_bytes) + " bytes, not " +
                                       std::to_string(nbytes));
  if (!mailbox || !aligned(mailbox, 16))
    return fail(MXFP8_ERR_INVALID, "mailbox must be a 16-byte aligned device pointer");
  if (!state || !aligned(state, 16))
    return fail(MXFP8_ERR_INVALID, "state must be a 16-byte aligned device int32[4]");
  if (!in || !aligned(in, 16) || !out || !aligned(out, 16))
    return fail(MXFP8_ERR_INVALID, "in and out must be 16-byte aligned device pointers");
  cudaError_t e = launch_lamport_gather(in, out, mailbox, state, capacity_bytes, nbytes,
                                        timeout_ns ? timeout_ns : kDefaultPollTimeoutNs,
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "launching the gather");
  return MXFP8_OK;
}

mxfp8_status mxfp8_mailbox_status(const int32_t* stage_state, int32_t* words, void* stream) {
  if (!stage_state || !words) return fail(MXFP8_ERR_INVALID, "stage_state and words are required");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(words, stage_state, 4 * sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "reading the state words");
  if (words[3] & (MXFP8_FLAG_POLL_TIMEOUT | MXFP8_FLAG_GEMM_TIMEOUT))
    return fail(MXFP8_ERR_TIMEOUT, "a device-side wait ran out of time (flags " +
                                       std::to_string(words[3]) + ")");
  if ((words[3] & MXFP8_FLAG_BAD_STATE) || words[0] < 0 || words[0] >= MXFP8_MAILBOX_GENERATIONS ||
      words[1] < 0 || words[1] >= MXFP8_MAILBOX_GENERATIONS)
    return fail(MXFP8_ERR_STATE, "the state words hold a generation outside 0..2");
  return MXFP8_OK;
}

void mxfp8_publish_gemm_destroy(mxfp8_publish_gemm* gemm) { delete gemm; }

}  // extern "C"

// ------------------------------------------------ the allocation-free call
// For callers that cannot allocate device memory: W's re-laid scale chunks go
// into this file-scope array instead of a caller-provided workspace.  Its
// name is a host-side stand-in in host code, so host code uses only the
// device address resolved below, once per device, with that device current.
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[MXFP8_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
uint8_t* g_noalloc_address[kMaxDevices] = {};

mxfp8_status noalloc_scratch(int device, uint8_t** out) {
  if (device < 0 || device >= kMaxDevices)
    return fail(MXFP8_ERR_UNSUPPORTED, "device ordinal out of range for the scratch table");
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_address[device] == nullptr) {
    void* address = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&address, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch array)");
    g_noalloc_address[device] = static_cast<uint8_t*>(address);
  }
  *out = g_noalloc_address[device];
  return MXFP8_OK;
}

// The set-up of an allocation-free call that depends only on the weight's
// address and the descriptor (kept per device from the last call), plus the
// activations' tensor map, kept while x and m repeat.
struct NoallocPlan {
  mxfp8_gemm_desc desc;  // resolved tactic
  int k_tiles;
  int tiles_per_split;
  TmemPlan tmem;
  GemmSmemLayout layout;
  CUtensorMap tmap_w;
  const void* x;
  int m;
  int32_t x_pieces;
  CUtensorMap tmap_x;
};

LastRequestCache<NoallocPlan, kMaxDevices> g_noalloc_plans;

}  // namespace

extern "C" mxfp8_status mxfp8_publish_gemm_run_noalloc(const mxfp8_gemm_desc* desc, const void* w,
                                                       const void* w_scale, const void* x,
                                                       const void* x_scale, int32_t m, void* c,
                                                       void* mailbox, int32_t* stage_state,
                                                       void* stream) {
  mxfp8_status st = check_desc(desc);
  if (st != MXFP8_OK) return st;
  if (desc->w_layout == MXFP8_W_TILED)
    return fail(MXFP8_ERR_UNSUPPORTED, "the allocation-free call reads W in place (no tiled copy)");
  if (!w || !aligned(w, 16)) return fail(MXFP8_ERR_INVALID, "w must be a 16-byte aligned device pointer");
  if (!w_scale) return fail(MXFP8_ERR_INVALID, "w_scale is NULL");
  st = check_mailbox(mailbox, stage_state, desc->capacity_m, desc->n);
  if (st != MXFP8_OK) return st;
  const int limit = std::min(MXFP8_MAX_ROWS, static_cast<int>(desc->capacity_m));
  if (m < 1 || m > limit)
    return fail(MXFP8_ERR_UNSUPPORTED,
                "m must be in 1.." + std::to_string(limit) + ", got " + std::to_string(m));
  if (!x || !aligned(x, 16)) return fail(MXFP8_ERR_INVALID, "x must be a 16-byte aligned device pointer");
  if (!x_scale) return fail(MXFP8_ERR_INVALID, "x_scale is NULL");
  if (c && !aligned(c, 16)) return fail(MXFP8_ERR_INVALID, "c must be 16-byte aligned");
  const size_t need = scale_chunk_bytes(desc->n, desc->k, sizing_fold(desc->fold));
  if (need > MXFP8_NOALLOC_SCRATCH_BYTES)
    return fail(MXFP8_ERR_UNSUPPORTED,
                "N=" + std::to_string(desc->n) + ", K=" + std::to_string(desc->k) + " needs " +
                    std::to_string(need) + " scratch bytes; the allocation-free call holds " +
                    std::to_string(MXFP8_NOALLOC_SCRATCH_BYTES));

  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  uint8_t* scratch = nullptr;
  st = noalloc_scratch(device, &scratch);
  if (st != MXFP8_OK) return st;

  // Resolving the tactic, encoding W's tensor map and raising the kernel's
  // shared-memory limit happen once per (device, w, descriptor); x's map once
  // per (x, m).
  NoallocPlan plan;
  auto make = [&](NoallocPlan* pl) {
    mxfp8_gemm_desc d = *desc;
    d.w_layout = MXFP8_W_IN_PLACE;
    DeviceLimits lim;
    mxfp8_status s2 = device_limits(device, &lim);
    if (s2 != MXFP8_OK) return s2;
    s2 = resolve_tactic(&d, lim);
    if (s2 != MXFP8_OK) return s2;
    pl->desc = d;
    pl->k_tiles = k_tiles_for_fold(d.k, d.fold);
    pl->tiles_per_split = (pl->k_tiles + d.split_k - 1) / d.split_k;
    pl->tmem = gemm_tmem_plan(d.stages, d.acc_blocks, d.fold, d.cta_k / kTileK);
    pl->layout = launch_layout(d, pl->tiles_per_split, lim);
    s2 = encode_rows(&pl->tmap_w, w, static_cast<uint64_t>(d.k), static_cast<uint64_t>(d.n),
                     kBlockN / d.fold);
    if (s2 != MXFP8_OK) return s2;
    pl->x = nullptr;
    pl->m = 0;
    return ensure_smem_attribute(device, d.split_k, d.fold, d.cta_k / kTileK,
                                 static_cast<int>(pl->layout.total), false);
  };
  auto refresh = [&](NoallocPlan* pl) {
    if (pl->x == x && pl->m == m) return MXFP8_OK;
    pl->x = nullptr;
    const mxfp8_status s2 = encode_x(&pl->tmap_x, x, pl->desc.k, m,
                                     pl->desc.fold * (pl->desc.cta_k / kTileK), &pl->x_pieces);
    if (s2 != MXFP8_OK) return s2;
    pl->x = x;
    pl->m = m;
    return MXFP8_OK;
  };
  st = g_noalloc_plans.get(device, NoallocRequest{w, *desc}, &plan, make, refresh);
  if (st != MXFP8_OK) return st;

  const mxfp8_gemm_desc& d = plan.desc;
  GemmParams p{};
  p.n = d.n;
  p.k = d.k;
  p.m = m;
  p.k_tiles = plan.k_tiles;
  p.tiles_per_split = plan.tiles_per_split;
  p.stages = d.stages;
  p.capacity = d.capacity_m;
  p.publish = 1;
  p.acc_blocks = d.acc_blocks;
  p.l2_prefetch = std::max(0, static_cast<int>(d.l2_prefetch));
  p.l2_prefetch_early = std::max(0, static_cast<int>(d.l2_prefetch_early));
  p.early_ctas = early_ctas_of(d);
  p.pipes = d.pipes;
  p.tmem_load = d.tmem_load;
  p.fold = d.fold;
  p.x_pieces = plan.x_pieces;
  p.tiles_per_stage = d.cta_k / kTileK;
  p.tmem = plan.tmem;
  p.x_scale = static_cast<const uint8_t*>(x_scale);
  p.w_sf = scratch;
  p.w_tiled = nullptr;
  p.c = static_cast<uint16_t*>(c);
  p.mailbox = static_cast<uint16_t*>(mailbox);
  p.state = stage_state;
  p.wait_limit_ns = static_cast<uint64_t>(d.wait_limit_ms) * 1000000ull;
  p.smem = plan.layout;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  e = launch_relayout_w_scales(static_cast<const uint8_t*>(w_scale), scratch, d.n, d.k, d.fold, s);
  if (e != cudaSuccess) return cuda_fail(e, "launching the W scale re-layout");
  // The re-layout right before it writes the scale chunks the GEMM's producer
  // reads before its grid wait, so this launch takes a full stream dependency.
  e = launch_publish_gemm(plan.tmap_w, plan.tmap_x, p, d.split_k, s, false);
  if (e != cudaSuccess) return cuda_fail(e, "launching the publishing GEMM");
  return MXFP8_OK;
}

extern "C" {

const char* mxfp8_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
