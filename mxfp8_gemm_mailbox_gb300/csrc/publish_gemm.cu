// MXFP8 low-batch GEMM with a publishing epilogue, for sm_103a.
//
// C[t][n] = sum_k W[n][k] x[t][k] (page "vllm.models.deepseek_v41.nvidia.
// specialized_decode.boundary.publishing_gemm", module description "GEMM
// structure"): the weight is the MMA's A operand (128 output columns per CTA,
// N/128 tiles), the at most 8 activation rows its B operand (N = 8).  Each
// CTA of a split-K cluster of S multiplies one K slice; the FP32 partials are
// exchanged through distributed shared memory and each CTA reduces 1/S of
// the tokens.  The epilogue rounds to BF16, writes C, and publishes every
// value with negative zero cleared into generation stage_state[0] of the
// mailbox as aligned 16-byte packs of eight consecutive columns, then one
// thread sets stage_state[1] (same page, publish_value and epilog_warp).
//
// Warp roles (192 threads):
//   warp 0      TMA producer: W tile + W scale chunk per stage (started
//               before the programmatic grid wait), x tile (after it).
//   warp 1      tensor-memory allocation; one thread issues tcgen05.cp of the
//               W scales and the block-scaled tcgen05.mma per 32-wide K block.
//   warps 2-5   epilogue: x scales into tensor memory, accumulator read-back
//               (tcgen05.ld 32x32b: thread = output column, 8 registers =
//               8 tokens), split-K exchange, BF16 rounding, C store, publish.
//
// Tensor-memory columns: [0, 8) FP32 accumulator (lane = output column,
// column = token); [sfa_col, +4*stages) the W scale ring and [sfb_col,
// +4*stages) the x scale ring, one 4-column slot per stage each, filled by
// tcgen05.cp (32x128b, multicast to the four lane quarters) from 16-byte-row
// scale chunks in shared memory.  Every scale address is 4-column aligned.
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace mxfp8 {
namespace {

constexpr uint32_t kStageTxBytes = kWTileBytes + kXTileBytes + kSfChunkBytes;

// Instruction descriptor of kind::mxf8f6f4 with block scaling: A and B E4M3
// (format 0), both K-major, N = 8 (bits 17-22: N >> 3), E8M0 scales (bit 23),
// M = 128 (bits 24-28: M >> 4).  The scale-factor byte ids of A (bits 29-30)
// and B (bits 4-5) select the K block inside a 32-bit scale column.
constexpr uint32_t kIdescBase =
    (static_cast<uint32_t>(kRows >> 3) << 17) | (1u << 23) | (static_cast<uint32_t>(kBlockN >> 4) << 24);

__device__ __forceinline__ uint32_t idesc_for_block(uint32_t kb) {
  return kIdescBase | (kb << 4) | (kb << 29);
}

// Each BF16 half equal to 0x8000 becomes 0x0000, so no word is the sentinel.
__device__ __forceinline__ uint32_t clear_negative_zero(uint32_t w) {
  uint32_t lo = w & 0xFFFFu, hi = w >> 16;
  lo = (lo == 0x8000u) ? 0u : lo;
  hi = (hi == 0x8000u) ? 0u : hi;
  return lo | (hi << 16);
}

__device__ __forceinline__ void raise_flag(int32_t* state, uint32_t bit) {
  atomicOr(reinterpret_cast<unsigned int*>(state + 3), bit);
}

__device__ __forceinline__ void epilogue_barrier() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// acc[index] for a runtime index without spilling the array to local memory.
template <int N>
__device__ __forceinline__ float select(const float (&acc)[N], int index) {
  float v = acc[0];
#pragma unroll
  for (int q = 1; q < N; ++q) v = (q == index) ? acc[q] : v;
  return v;
}

__device__ __forceinline__ uint16_t bf16_bits_rn(float v) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

template <int S>
__global__ void __launch_bounds__(kThreads, 1)
    publish_gemm_kernel(const __grid_constant__ CUtensorMap tmap_w,
                        const __grid_constant__ CUtensorMap tmap_x,
                        const __grid_constant__ GemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_addr(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = ptx::smem_addr(smem);
  const GemmSmemLayout& L = p.smem;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t split = (S > 1) ? ptx::cluster_ctarank() : 0u;
  const int tile = blockIdx.x / S;
  const int kt_begin = static_cast<int>(split) * p.tiles_per_split;
  const int kt_end = min(p.k_tiles, kt_begin + p.tiles_per_split);
  const int nkt = max(0, kt_end - kt_begin);
  const int stages = p.stages;

  const uint32_t bar_full = sbase + L.bars;
  const uint32_t bar_empty = bar_full + 8u * stages;
  const uint32_t bar_acc = bar_empty + 8u * stages;
  const uint32_t bar_sfb = bar_acc + 8u;
  const uint32_t bar_recv = bar_sfb + 8u;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L.misc);  // [0] tmem base, [1] generation

  if (tid == 0) {
    ptx::prefetch_tensormap(&tmap_w);
    ptx::prefetch_tensormap(&tmap_x);
    for (int s = 0; s < stages; ++s) {
      ptx::mbar_init(bar_full + 8u * s, 1);
      ptx::mbar_init(bar_empty + 8u * s, 1);
    }
    ptx::mbar_init(bar_acc, 1);
    ptx::mbar_init(bar_sfb, 128);
    ptx::mbar_init(bar_recv, 1);
    ptx::fence_mbarrier_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(sbase + L.misc, p.tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  if (S > 1) {
    ptx::cluster_sync();  // peers' barriers exist before any remote store
  } else {
    __syncthreads();
  }
  ptx::tc_fence_after();
  const uint32_t tmem = misc[0];

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      ptx::launch_dependents();
      const uint64_t pol_stream = ptx::policy_evict_first();
      const uint64_t pol_keep = ptx::policy_evict_last();
      const int npre = min(stages, nkt);
      // W and its scales do not depend on the previous kernel: start them now.
      for (int i = 0; i < npre; ++i) {
        const uint32_t full = bar_full + 8u * i;
        const int kt = kt_begin + i;
        ptx::mbar_arrive_expect_tx(full, kStageTxBytes);
        ptx::tma_load_2d(sbase + L.w + i * kWTileBytes, &tmap_w, kt * kTileK, tile * kBlockN, full,
                         pol_stream);
        ptx::bulk_load(sbase + L.sfa + i * kSfChunkBytes,
                       p.w_sf + (static_cast<size_t>(tile) * p.k_tiles + kt) * kSfChunkBytes,
                       kSfChunkBytes, full, pol_stream);
      }
      // The activations follow the programmatic grid wait.
      ptx::grid_dependency_wait();
      for (int i = 0; i < npre; ++i)
        ptx::tma_load_2d(sbase + L.x + i * kXTileBytes, &tmap_x, (kt_begin + i) * kTileK, 0,
                         bar_full + 8u * i, pol_keep);
      int issued = npre;
      for (int i = npre; i < nkt; ++i) {
        const int s = i % stages;
        const uint32_t use = static_cast<uint32_t>(i / stages);
        if (!ptx::mbar_wait(bar_empty + 8u * s, (use - 1u) & 1u, p.wait_limit_ns)) {
          raise_flag(p.state, 0x2u);
          break;
        }
        const uint32_t full = bar_full + 8u * s;
        const int kt = kt_begin + i;
        ptx::mbar_arrive_expect_tx(full, kStageTxBytes);
        ptx::tma_load_2d(sbase + L.w + s * kWTileBytes, &tmap_w, kt * kTileK, tile * kBlockN, full,
                         pol_stream);
        ptx::bulk_load(sbase + L.sfa + s * kSfChunkBytes,
                       p.w_sf + (static_cast<size_t>(tile) * p.k_tiles + kt) * kSfChunkBytes,
                       kSfChunkBytes, full, pol_stream);
        ptx::tma_load_2d(sbase + L.x + s * kXTileBytes, &tmap_x, kt * kTileK, 0, full, pol_keep);
        issued = i + 1;
      }
      // Copies still in flight land before the CTA leaves (immediate when the
      // MMA consumed them, which is the normal case).
      for (int i = max(0, issued - stages); i < issued; ++i)
        ptx::mbar_wait(bar_full + 8u * (i % stages), static_cast<uint32_t>(i / stages) & 1u,
                       p.wait_limit_ns);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      ptx::grid_dependency_wait();
      bool ok = true;
      if (nkt > 0) {
        ok = ptx::mbar_wait(bar_sfb, 0, p.wait_limit_ns);
        if (!ok) raise_flag(p.state, 0x2u);
        ptx::tc_fence_after();
      }
      const uint32_t d_tmem = tmem;  // accumulator at column 0
      for (int i = 0; i < nkt && ok; ++i) {
        const int s = i % stages;
        if (!ptx::mbar_wait(bar_full + 8u * s, static_cast<uint32_t>(i / stages) & 1u,
                            p.wait_limit_ns)) {
          raise_flag(p.state, 0x2u);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t sfa_t = tmem + p.sfa_col + 4u * s;
        const uint32_t sfb_t = tmem + p.sfb_col + 4u * s;
        ptx::tmem_cp_32x128b_warpx4(sfa_t, ptx::desc_rows16(sbase + L.sfa + s * kSfChunkBytes));
        ptx::tmem_cp_32x128b_warpx4(sfb_t, ptx::desc_rows16(sbase + L.sx + i * 128));
        const uint32_t a0 = sbase + L.w + s * kWTileBytes;
        const uint32_t b0 = sbase + L.x + s * kXTileBytes;
#pragma unroll
        for (uint32_t kb = 0; kb < kSfPerTile; ++kb) {
          ptx::mma_mxf8(d_tmem, ptx::desc_kmajor_sw128(a0 + 32u * kb),
                        ptx::desc_kmajor_sw128(b0 + 32u * kb), idesc_for_block(kb),
                        (i > 0 || kb > 0) ? 1u : 0u, sfa_t, sfb_t);
        }
        ptx::mma_commit(bar_empty + 8u * s);
      }
      if (nkt > 0 && ok)
        ptx::mma_commit(bar_acc);
      else
        ptx::mbar_arrive(bar_acc);
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int etid = tid - 64;               // 0..127
    const int quarter = warp & 3;            // the 32 TMEM lanes this warp reaches
    const int col = quarter * 32 + lane;     // output column within the tile
    const uint32_t lane_base = static_cast<uint32_t>(quarter * 32) << 16;
    ptx::grid_dependency_wait();
    if (etid == 0) misc[1] = ptx::ld_volatile_u32(p.state + 0);

    // x scales of this CTA's K range as one 128-byte chunk per K tile: row r
    // (< 8) of tile j at byte j * 128 + r * 16, its four E8M0 codes first.
    // Rows >= m and blocks past K take 127 (a scale of 1; those x elements
    // are zero).  The copy of a chunk reads 32 rows; rows 8..31 (the next
    // chunks, or the zero tail) feed no output column.
    uint8_t* sx = smem + L.sx;
    const int kblocks = p.k / 32;
    const int sx_bytes = p.tiles_per_split * 128 + 384;
    for (int b = etid; b < sx_bytes; b += 128) {
      const int j = b / 128;
      const int r = (b % 128) / 16;
      const int q = b % 16;
      uint8_t v = 0;
      if (q < kSfPerTile && j < nkt) {
        const int kb = (kt_begin + j) * kSfPerTile + q;
        v = 127;
        if (r < p.m && kb < kblocks) v = p.x_scale[static_cast<size_t>(r) * kblocks + kb];
      }
      sx[b] = v;
    }
    ptx::fence_proxy_async_smem();  // the tensor-memory copy reads them
    ptx::mbar_arrive(bar_sfb);

    if (!ptx::mbar_wait(bar_acc, 0, p.wait_limit_ns)) raise_flag(p.state, 0x2u);
    ptx::tc_fence_after();
    float acc[kRows];
    if (nkt > 0) {
      uint32_t r[8];
      ptx::tmem_ld_32x32b_x8(tmem + lane_base, r);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int q = 0; q < kRows; ++q) acc[q] = __uint_as_float(r[q]);
    } else {
      // A split with no K tiles contributes zeros.
#pragma unroll
      for (int q = 0; q < kRows; ++q) acc[q] = 0.0f;
    }

    constexpr int kShard = kRows / S;  // tokens this CTA reduces and stores
    float owned[kShard];
    if constexpr (S > 1) {
      if (etid == 0)
        ptx::mbar_arrive_expect_tx(bar_recv, static_cast<uint32_t>((S - 1) * kShard * kBlockN * 4));
#pragma unroll
      for (int peer = 0; peer < S; ++peer) {
        if (peer == static_cast<int>(split)) continue;
        const int sender = static_cast<int>(split) < peer ? static_cast<int>(split)
                                                          : static_cast<int>(split) - 1;
        const uint32_t remote_bar = ptx::map_to_rank(bar_recv, peer);
#pragma unroll
        for (int jj = 0; jj < kShard; ++jj) {
          const uint32_t local = sbase + L.recv + ((sender * kShard + jj) * kBlockN + col) * 4;
          ptx::st_async_remote(ptx::map_to_rank(local, peer),
                               __float_as_uint(acc[peer * kShard + jj]), remote_bar);
        }
      }
      if (!ptx::mbar_wait_cluster(bar_recv, 0, p.wait_limit_ns)) raise_flag(p.state, 0x2u);
      const float* recv = reinterpret_cast<const float*>(smem + L.recv);
#pragma unroll
      for (int jj = 0; jj < kShard; ++jj) {
        float total = 0.0f;
#pragma unroll
        for (int src = 0; src < S; ++src) {
          float v;
          if (src == static_cast<int>(split)) {
            v = select(acc, static_cast<int>(split) * kShard + jj);
          } else {
            const int sidx = src < static_cast<int>(split) ? src : src - 1;
            v = recv[(sidx * kShard + jj) * kBlockN + col];
          }
          total = (src == 0) ? v : total + v;  // K-slice order, on every CTA
        }
        owned[jj] = total;
      }
    } else {
#pragma unroll
      for (int jj = 0; jj < kShard; ++jj) owned[jj] = acc[jj];
    }

    uint16_t* ctile = reinterpret_cast<uint16_t*>(smem + L.ctile);  // [kShard][128]
#pragma unroll
    for (int jj = 0; jj < kShard; ++jj) ctile[jj * kBlockN + col] = bf16_bits_rn(owned[jj]);
    epilogue_barrier();

    const uint32_t g = misc[1];
    const bool generation_ok = g < static_cast<uint32_t>(kGenerations);
    const size_t n0 = static_cast<size_t>(tile) * kBlockN;
    for (int pk = etid; pk < kShard * (kBlockN / 8); pk += 128) {
      const int jj = pk / (kBlockN / 8);
      const int chunk = pk % (kBlockN / 8);
      const int t = static_cast<int>(split) * kShard + jj;
      if (t >= p.m) continue;
      const uint4 v = *reinterpret_cast<const uint4*>(ctile + jj * kBlockN + chunk * 8);
      const size_t column = n0 + chunk * 8;
      if (p.c != nullptr) ptx::st_v4(p.c + static_cast<size_t>(t) * p.n + column, v);
      if (p.publish && generation_ok) {
        const uint4 clean = make_uint4(clear_negative_zero(v.x), clear_negative_zero(v.y),
                                       clear_negative_zero(v.z), clear_negative_zero(v.w));
        ptx::st_v4(p.mailbox + (static_cast<size_t>(g) * p.capacity + t) * p.n + column, clean);
      }
    }
    // Hand the generation to the consumer, once per grid.
    if (p.publish && blockIdx.x == 0 && etid == 0) {
      if (generation_ok)
        p.state[1] = static_cast<int32_t>(g);
      else
        raise_flag(p.state, 0x4u);
    }
  }

  // --------------------------------------------------------------- teardown
  ptx::tc_fence_before();
  __syncthreads();
  if (S > 1) {
    __syncwarp();
    ptx::cluster_sync();  // no CTA leaves while a peer may still address it
  }
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, p.tmem_cols);
  }
}

// W scales [n][k/32] -> [n/128][k_tiles][512]: inside a chunk, row r of the
// tile and K block b of the stage sit at byte (r % 32) * 16 + (r / 32) * 4 + b,
// the order the 32x128b tensor-memory copy and the MMA's scale lookup expect.
// Blocks past K take 127.
__global__ void relayout_w_scales_kernel(const uint8_t* __restrict__ w_scale,
                                         uint8_t* __restrict__ w_sf, int n, int kblocks,
                                         int k_tiles) {
  const size_t total = static_cast<size_t>(n / kBlockN) * k_tiles * kSfChunkBytes;
  for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t chunk = idx / kSfChunkBytes;
    const int within = static_cast<int>(idx % kSfChunkBytes);
    const int tile = static_cast<int>(chunk / k_tiles);
    const int kt = static_cast<int>(chunk % k_tiles);
    const int r0 = within / 16;
    const int r1 = (within % 16) / 4;
    const int b = within % 4;
    const int row = tile * kBlockN + r1 * 32 + r0;
    const int blk = kt * kSfPerTile + b;
    w_sf[idx] = blk < kblocks ? w_scale[static_cast<size_t>(row) * kblocks + blk] : 127;
  }
}

template <int S>
cudaError_t launch_impl(const CUtensorMap& tmap_w, const CUtensorMap& tmap_x, const GemmParams& p,
                        cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((p.n / kBlockN) * S), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = p.smem.total;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  int count = 0;
  attrs[count].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[count].val.programmaticStreamSerializationAllowed = 1;
  ++count;
  if (S > 1) {
    attrs[count].id = cudaLaunchAttributeClusterDimension;
    attrs[count].val.clusterDim.x = S;
    attrs[count].val.clusterDim.y = 1;
    attrs[count].val.clusterDim.z = 1;
    ++count;
  }
  cfg.attrs = attrs;
  cfg.numAttrs = count;
  return cudaLaunchKernelEx(&cfg, publish_gemm_kernel<S>, tmap_w, tmap_x, p);
}

}  // namespace

GemmSmemLayout gemm_smem_layout(int stages, int split_k, int tiles_per_split) {
  GemmSmemLayout L{};
  L.w = 0;
  L.x = L.w + stages * kWTileBytes;
  L.sfa = L.x + stages * kXTileBytes;
  L.ctile = L.sfa + stages * kSfChunkBytes;
  L.recv = L.ctile + kRows * kBlockN * 2;
  const uint32_t recv_bytes =
      split_k > 1 ? static_cast<uint32_t>((split_k - 1) * (kRows / split_k) * kBlockN * 4) : 0u;
  L.sx = L.recv + recv_bytes;
  const uint32_t sx_bytes = static_cast<uint32_t>(tiles_per_split * 128 + 384);
  L.bars = (L.sx + sx_bytes + 7u) & ~7u;
  L.misc = L.bars + static_cast<uint32_t>(2 * stages + 3) * 8u;
  L.total = L.misc + 16u + 1024u;
  return L;
}

uint32_t gemm_tmem_columns(int stages, int tiles_per_split, uint32_t* sfb_col, uint32_t* sfa_col) {
  (void)tiles_per_split;
  const uint32_t sfa = 8u;
  const uint32_t sfb = sfa + 4u * static_cast<uint32_t>(stages);
  const uint32_t used = sfb + 4u * static_cast<uint32_t>(stages);
  uint32_t cols = 32;
  while (cols < used) cols <<= 1;
  if (sfb_col) *sfb_col = sfb;
  if (sfa_col) *sfa_col = sfa;
  return cols;
}

cudaError_t set_gemm_smem_attribute(int split_k, int bytes) {
  switch (split_k) {
    case 1:
      return cudaFuncSetAttribute(publish_gemm_kernel<1>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    case 2:
      return cudaFuncSetAttribute(publish_gemm_kernel<2>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    case 4:
      return cudaFuncSetAttribute(publish_gemm_kernel<4>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_publish_gemm(const CUtensorMap& tmap_w, const CUtensorMap& tmap_x,
                                const GemmParams& p, int split_k, cudaStream_t stream) {
  switch (split_k) {
    case 1:
      return launch_impl<1>(tmap_w, tmap_x, p, stream);
    case 2:
      return launch_impl<2>(tmap_w, tmap_x, p, stream);
    case 4:
      return launch_impl<4>(tmap_w, tmap_x, p, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t launch_relayout_w_scales(const uint8_t* w_scale, uint8_t* w_sf, int n, int k,
                                     cudaStream_t stream) {
  const int k_tiles = (k + kTileK - 1) / kTileK;
  const size_t total = static_cast<size_t>(n / kBlockN) * k_tiles * kSfChunkBytes;
  const int threads = 256;
  const int blocks = static_cast<int>(std::min<size_t>((total + threads - 1) / threads, 4096));
  relayout_w_scales_kernel<<<blocks, threads, 0, stream>>>(w_scale, w_sf, n, k / 32, k_tiles);
  return cudaGetLastError();
}

}  // namespace mxfp8
