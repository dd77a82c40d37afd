// The tagged-pair mailbox (page "vllm.models.deepseek_v41.amd.mono.common.
// sync", Mailbox: every 32-bit value stored next to the launch's tag; a
// consumer polls the payload until all tags match; nothing is reset), as a
// protocol for the decode projection's output on sm_103a.
//
// pairs[t][w] = (word, tag), word w holding BF16 columns 2w (low half) and
// 2w + 1.  One thread per 16-byte pack of C (eight columns = four words)
// writes two 16-byte stores {w0, tag, w1, tag}, {w2, tag, w3, tag}, so each
// value travels in the same store as its tag.  The bits move unchanged: no
// sentinel, hence no negative-zero clearing and no reset store.
#include <algorithm>

#include "internal.h"
#include "ptx.cuh"

namespace mxfp8 {
namespace {

constexpr int kTaggedThreads = 128;

__global__ void tagged_init_kernel(uint4* __restrict__ pairs, size_t count) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < count;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    pairs[i] = make_uint4(0u, 0u, 0u, 0u);
}

__global__ void __launch_bounds__(kTaggedThreads)
    tagged_publish_kernel(uint4* __restrict__ pairs, int n, int m,
                          const uint16_t* __restrict__ c, uint32_t tag) {
  ptx::launch_dependents();
  ptx::grid_dependency_wait();
  const int packs_per_row = n / 8;
  const int pack = blockIdx.x * kTaggedThreads + threadIdx.x;
  if (pack >= m * packs_per_row) return;
  const int t = pack / packs_per_row;
  const int c8 = pack % packs_per_row;
  const uint4 v = *reinterpret_cast<const uint4*>(c + static_cast<size_t>(t) * n + c8 * 8);
  uint4* dst = pairs + 2 * (static_cast<size_t>(t) * packs_per_row + c8);
  ptx::st_v4(dst, make_uint4(v.x, tag, v.y, tag));
  ptx::st_v4(dst + 1, make_uint4(v.z, tag, v.w, tag));
}

__global__ void __launch_bounds__(kTaggedThreads)
    tagged_consume_kernel(const uint4* __restrict__ pairs, int n, int m, uint32_t tag,
                          uint16_t* __restrict__ out, uint64_t timeout_ns, int32_t* flags) {
  ptx::launch_dependents();
  ptx::grid_dependency_wait();
  const int packs_per_row = n / 8;
  const int pack = blockIdx.x * kTaggedThreads + threadIdx.x;
  if (pack >= m * packs_per_row) return;
  const int t = pack / packs_per_row;
  const int c8 = pack % packs_per_row;
  const uint4* src = pairs + 2 * (static_cast<size_t>(t) * packs_per_row + c8);
  uint4 a = ptx::ld_volatile_v4(src);
  uint4 b = ptx::ld_volatile_v4(src + 1);
  if (a.y != tag || a.w != tag || b.y != tag || b.w != tag) {
    const uint64_t start = ptx::globaltimer();
    for (;;) {
      a = ptx::ld_volatile_v4(src);
      b = ptx::ld_volatile_v4(src + 1);
      if (a.y == tag && a.w == tag && b.y == tag && b.w == tag) break;
      if (ptx::globaltimer() - start > timeout_ns) {
        if (flags != nullptr) atomicOr(reinterpret_cast<unsigned int*>(flags), 0x1u);
        break;
      }
    }
  }
  ptx::st_v4(out + static_cast<size_t>(t) * n + c8 * 8, make_uint4(a.x, a.z, b.x, b.z));
}

cudaLaunchConfig_t pdl_config(int packs, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((packs + kTaggedThreads - 1) / kTaggedThreads), 1, 1);
  cfg.blockDim = dim3(kTaggedThreads, 1, 1);
  cfg.stream = stream;
  attr->id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr->val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

}  // namespace

cudaError_t launch_tagged_init(void* pairs, size_t bytes, cudaStream_t stream) {
  const size_t count = bytes / 16;
  const int threads = 256;
  const int blocks =
      static_cast<int>(std::max<size_t>(1, std::min<size_t>((count + threads - 1) / threads, 1024)));
  tagged_init_kernel<<<blocks, threads, 0, stream>>>(static_cast<uint4*>(pairs), count);
  return cudaGetLastError();
}

cudaError_t launch_tagged_publish(void* pairs, int n, int m, const uint16_t* c, uint32_t tag,
                                  cudaStream_t stream) {
  cudaLaunchAttribute attr;
  cudaLaunchConfig_t cfg = pdl_config(m * (n / 8), stream, &attr);
  return cudaLaunchKernelEx(&cfg, tagged_publish_kernel, static_cast<uint4*>(pairs), n, m, c, tag);
}

cudaError_t launch_tagged_consume(const void* pairs, int n, int m, uint32_t tag, uint16_t* out,
                                  uint64_t timeout_ns, int32_t* flags, cudaStream_t stream) {
  cudaLaunchAttribute attr;
  cudaLaunchConfig_t cfg = pdl_config(m * (n / 8), stream, &attr);
  return cudaLaunchKernelEx(&cfg, tagged_consume_kernel, static_cast<const uint4*>(pairs), n, m,
                            tag, out, timeout_ns, flags);
}

}  // namespace mxfp8
