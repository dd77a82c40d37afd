// The Lamport all-gather with one rank (page "vllm.models.deepseek_v41.
// nvidia.ops.cute_dsl.all_gather", module description steps 1-3 and
// _AllGatherKernel.kernel), on its own mailbox: mailbox[generation][pack] of
// 16-byte packs, three generations of `capacity` bytes, and state words [0]
// the call's generation, [1] the arrival count ([2] unused, [3] error flags).
//
// One thread per 16-byte pack: publish the pack into this rank's slot of the
// generation with every word equal to the sentinel 0x80000000 cleared to 0;
// trigger the dependents; poll the slot (the rank's own, the only one) until
// no word is the sentinel; write it to the output; store the sentinel back.
// Each CTA reads the generation once, before it counts itself in; the last
// CTA to arrive advances the generation and clears the count.
#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace mxfp8 {
namespace {

constexpr int kGatherThreads = 128;

__device__ __forceinline__ void raise_flag(int32_t* state, uint32_t bit) {
  atomicOr(reinterpret_cast<unsigned int*>(state + 3), bit);
}

__device__ __forceinline__ bool has_sentinel(const uint4& v) {
  return v.x == kSentinel || v.y == kSentinel || v.z == kSentinel || v.w == kSentinel;
}

__device__ __forceinline__ uint32_t clear_sentinel(uint32_t w) { return w == kSentinel ? 0u : w; }

__global__ void lamport_gather_init_kernel(uint4* __restrict__ mailbox, size_t packs,
                                           int32_t* __restrict__ state) {
  const uint4 sentinel = make_uint4(kSentinel, kSentinel, kSentinel, kSentinel);
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < packs;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    mailbox[i] = sentinel;
  if (blockIdx.x == 0 && threadIdx.x < 4) state[threadIdx.x] = 0;
}

__global__ void __launch_bounds__(kGatherThreads)
    lamport_gather_kernel(const uint4* __restrict__ in, uint4* __restrict__ out,
                          uint4* __restrict__ mailbox, int32_t* __restrict__ state,
                          int capacity_packs, int packs, uint64_t timeout_ns) {
  __shared__ uint32_t shared_generation;
  ptx::grid_dependency_wait();
  if (threadIdx.x == 0) {
    const uint32_t g = ptx::ld_volatile_u32(state + 0);
    shared_generation = g;
    if (ptx::atom_add_acq_rel(state + 1, 1u) == gridDim.x - 1) {
      if (g < static_cast<uint32_t>(kGenerations))
        state[0] = static_cast<int32_t>((g + 1u) % kGenerations);
      else
        raise_flag(state, 0x4u);
      state[1] = 0;
    }
  }
  __syncthreads();
  const uint32_t g = shared_generation;
  if (g >= static_cast<uint32_t>(kGenerations)) {
    ptx::launch_dependents();
    return;  // a corrupted generation word: address nothing
  }
  const int pack = blockIdx.x * kGatherThreads + threadIdx.x;
  const bool active = pack < packs;
  uint4* slot = mailbox + static_cast<size_t>(g) * capacity_packs + pack;
  if (active) {
    const uint4 v = in[pack];
    ptx::st_v4(slot, make_uint4(clear_sentinel(v.x), clear_sentinel(v.y), clear_sentinel(v.z),
                                clear_sentinel(v.w)));
  }
  ptx::launch_dependents();
  if (!active) return;
  // The rank's own slot too: the published pack must land before the reset.
  uint4 v = ptx::ld_volatile_v4(slot);
  if (has_sentinel(v)) {
    const uint64_t start = ptx::globaltimer();
    for (;;) {
      v = ptx::ld_volatile_v4(slot);
      if (!has_sentinel(v)) break;
      if (ptx::globaltimer() - start > timeout_ns) {
        raise_flag(state, 0x1u);
        break;
      }
    }
  }
  ptx::st_v4(out + pack, v);
  ptx::st_v4(slot, make_uint4(kSentinel, kSentinel, kSentinel, kSentinel));
}

}  // namespace

cudaError_t launch_lamport_gather_init(void* mailbox, int32_t* state, size_t capacity_bytes,
                                       cudaStream_t stream) {
  const size_t packs = static_cast<size_t>(kGenerations) * capacity_bytes / 16;
  const int threads = 256;
  const int blocks =
      static_cast<int>(std::max<size_t>(1, std::min<size_t>((packs + threads - 1) / threads, 1024)));
  lamport_gather_init_kernel<<<blocks, threads, 0, stream>>>(static_cast<uint4*>(mailbox), packs,
                                                             state);
  return cudaGetLastError();
}

cudaError_t launch_lamport_gather(const void* in, void* out, void* mailbox, int32_t* state,
                                  size_t capacity_bytes, size_t nbytes, uint64_t timeout_ns,
                                  cudaStream_t stream) {
  const int packs = static_cast<int>(nbytes / 16);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((packs + kGatherThreads - 1) / kGatherThreads), 1, 1);
  cfg.blockDim = dim3(kGatherThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, lamport_gather_kernel, static_cast<const uint4*>(in),
                            static_cast<uint4*>(out), static_cast<uint4*>(mailbox), state,
                            static_cast<int>(capacity_bytes / 16), packs, timeout_ns);
}

}  // namespace mxfp8
