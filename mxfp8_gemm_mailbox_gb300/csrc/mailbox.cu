// Lamport mailbox kernels: arm, consume, and the standalone publish of the
// unfused path.
//
// The protocol is the one of page "vllm.models.deepseek_v41.nvidia.ops.
// cute_dsl.all_gather" (module description, steps 1-3), with one rank: the
// mailbox holds three generations of 16-byte packs; an empty word is the
// sentinel 0x80000000; a consumer polls its slots until no word is the
// sentinel, copies them out and stores the sentinel back, and the generation
// advances.  The state words are [0] next generation, [1] active generation
// (page "vllm.models.deepseek_v41.nvidia.specialized_decode.boundary.
// publishing_gemm", module description), [2] zero (the all-gather counts its
// CTAs there; this consumer needs no count), [3] error flags.
#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace mxfp8 {
namespace {

constexpr int kConsumeThreads = 128;
constexpr uint32_t kFlagPollTimeout = 0x1u;
constexpr uint32_t kFlagBadState = 0x4u;

__device__ __forceinline__ void raise_flag(int32_t* state, uint32_t bit) {
  atomicOr(reinterpret_cast<unsigned int*>(state + 3), bit);
}

__device__ __forceinline__ bool has_sentinel(const uint4& v) {
  return v.x == kSentinel || v.y == kSentinel || v.z == kSentinel || v.w == kSentinel;
}

__device__ __forceinline__ uint32_t clear_negative_zero(uint32_t w) {
  uint32_t lo = w & 0xFFFFu, hi = w >> 16;
  lo = (lo == 0x8000u) ? 0u : lo;
  hi = (hi == 0x8000u) ? 0u : hi;
  return lo | (hi << 16);
}

// Every word of the mailbox becomes the sentinel; the state becomes zero.
__global__ void mailbox_init_kernel(uint4* __restrict__ mailbox, size_t packs,
                                    int32_t* __restrict__ state) {
  const uint4 sentinel = make_uint4(kSentinel, kSentinel, kSentinel, kSentinel);
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < packs;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    mailbox[i] = sentinel;
  if (blockIdx.x == 0 && threadIdx.x < 4) state[threadIdx.x] = 0;
}

// One thread per 16-byte pack of the m published rows.
__global__ void __launch_bounds__(kConsumeThreads)
    mailbox_consume_kernel(uint16_t* __restrict__ mailbox, int32_t* __restrict__ state,
                           int capacity, int n, int m, uint16_t* __restrict__ out,
                           uint64_t timeout_ns) {
  // The next kernel may launch now (its own grid wait covers this grid); the
  // GEMM (or publish kernel) before this one has completed and its stores
  // are visible after the grid wait.
  ptx::launch_dependents();
  ptx::grid_dependency_wait();
  // The active generation is written only by the publisher, so every thread
  // reads it, and loads its pack from all three generations alongside it
  // (one memory round trip instead of two), keeping the active one.  The
  // all-gather page's CTAs count themselves and the last one advances the
  // generation, because they read the word it advances; no CTA of this grid
  // reads the word it advances (state[0] is read by the next publisher, after
  // this grid completes), so one CTA advances it, with no count: a count
  // served CTA by CTA on one word measured 0.2 us a call on the N=4096,
  // K=4096 chain.
  const int packs_per_row = n / 8;
  const int pack = blockIdx.x * kConsumeThreads + threadIdx.x;
  const bool active = pack < m * packs_per_row;
  const int t = active ? pack / packs_per_row : 0;
  const int c8 = active ? pack % packs_per_row : 0;
  const size_t generation_stride = static_cast<size_t>(capacity) * n;
  uint16_t* slot0 = mailbox + static_cast<size_t>(t) * n + c8 * 8;
  const uint32_t g = ptx::ld_volatile_u32(state + 1);
  uint4 candidates[kGenerations];
  if (active) {
#pragma unroll
    for (int gg = 0; gg < kGenerations; ++gg)
      candidates[gg] = ptx::ld_volatile_v4(slot0 + gg * generation_stride);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (g < static_cast<uint32_t>(kGenerations)) {
      state[0] = static_cast<int32_t>((g + 1u) % kGenerations);
    } else {
      raise_flag(state, kFlagBadState);
    }
  }
  if (g >= static_cast<uint32_t>(kGenerations) || !active) return;

  uint16_t* slot = slot0 + g * generation_stride;
  uint4 v = g == 0 ? candidates[0] : (g == 1 ? candidates[1] : candidates[2]);
  if (has_sentinel(v)) {
    const uint64_t start = ptx::globaltimer();
    for (;;) {
      v = ptx::ld_volatile_v4(slot);
      if (!has_sentinel(v)) break;
      if (ptx::globaltimer() - start > timeout_ns) {
        raise_flag(state, kFlagPollTimeout);
        break;
      }
    }
  }
  ptx::st_v4(out + static_cast<size_t>(t) * n + c8 * 8, v);
  ptx::st_v4(slot, make_uint4(kSentinel, kSentinel, kSentinel, kSentinel));
}

// The unfused path's publish: C [m][n] -> mailbox[state[0]], negative zero
// cleared, then state[1] = state[0].
__global__ void __launch_bounds__(kConsumeThreads)
    mailbox_publish_kernel(uint16_t* __restrict__ mailbox, int32_t* __restrict__ state,
                           int capacity, int n, int m, const uint16_t* __restrict__ c) {
  ptx::launch_dependents();
  ptx::grid_dependency_wait();
  const uint32_t g = ptx::ld_volatile_u32(state + 0);
  const bool first = blockIdx.x == 0 && threadIdx.x == 0;
  if (g >= static_cast<uint32_t>(kGenerations)) {
    if (first) raise_flag(state, kFlagBadState);
    return;
  }
  const int packs_per_row = n / 8;
  const int pack = blockIdx.x * kConsumeThreads + threadIdx.x;
  if (pack < m * packs_per_row) {
    const int t = pack / packs_per_row;
    const int c8 = pack % packs_per_row;
    const uint4 v =
        *reinterpret_cast<const uint4*>(c + static_cast<size_t>(t) * n + c8 * 8);
    const uint4 clean = make_uint4(clear_negative_zero(v.x), clear_negative_zero(v.y),
                                   clear_negative_zero(v.z), clear_negative_zero(v.w));
    ptx::st_v4(mailbox + (static_cast<size_t>(g) * capacity + t) * n + c8 * 8, clean);
  }
  if (first) state[1] = static_cast<int32_t>(g);
}

cudaLaunchConfig_t pdl_config(int blocks, int threads, cudaStream_t stream,
                              cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  attr->id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr->val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

cudaError_t launch_mailbox_init(uint16_t* mailbox, int32_t* state, int capacity, int n,
                                cudaStream_t stream) {
  const size_t packs = static_cast<size_t>(kGenerations) * capacity * n / 8;
  const int threads = 256;
  const int blocks =
      static_cast<int>(std::max<size_t>(1, std::min<size_t>((packs + threads - 1) / threads, 1024)));
  mailbox_init_kernel<<<blocks, threads, 0, stream>>>(reinterpret_cast<uint4*>(mailbox), packs,
                                                      state);
  return cudaGetLastError();
}

cudaError_t launch_mailbox_consume(uint16_t* mailbox, int32_t* state, int capacity, int n, int m,
                                   uint16_t* out, uint64_t timeout_ns, cudaStream_t stream) {
  const int packs = m * (n / 8);
  const int blocks = (packs + kConsumeThreads - 1) / kConsumeThreads;
  cudaLaunchAttribute attr;
  cudaLaunchConfig_t cfg = pdl_config(blocks, kConsumeThreads, stream, &attr);
  return cudaLaunchKernelEx(&cfg, mailbox_consume_kernel, mailbox, state, capacity, n, m, out,
                            timeout_ns);
}

cudaError_t launch_mailbox_publish(uint16_t* mailbox, int32_t* state, int capacity, int n, int m,
                                   const uint16_t* c, cudaStream_t stream) {
  const int packs = m * (n / 8);
  const int blocks = (packs + kConsumeThreads - 1) / kConsumeThreads;
  cudaLaunchAttribute attr;
  cudaLaunchConfig_t cfg = pdl_config(blocks, kConsumeThreads, stream, &attr);
  return cudaLaunchKernelEx(&cfg, mailbox_publish_kernel, mailbox, state, capacity, n, m, c);
}

}  // namespace mxfp8
