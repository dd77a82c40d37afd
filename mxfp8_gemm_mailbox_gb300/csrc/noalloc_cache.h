// Host-side memo of the allocation-free call's set-up work.  That call takes
// no handle, so without a memo every call would re-resolve the tactic and
// re-encode the weight's tensor map; with it, a call that repeats the
// previous call's weight pointer and descriptor on the same device reuses
// what that call built.  Header-only and free of CUDA types, so the policy
// can be exercised on a host without a GPU.
#pragma once
#include <cstring>
#include <mutex>

#include "mxfp8_mailbox.h"

namespace mxfp8 {

// What identifies the set-up work: the weight's address and the descriptor
// exactly as the caller passed it (every field is an int32, so the struct
// has no padding and compares bytewise).
struct NoallocRequest {
  const void* w;
  mxfp8_gemm_desc desc;
};

inline bool same_request(const NoallocRequest& a, const NoallocRequest& b) {
  return a.w == b.w && std::memcmp(&a.desc, &b.desc, sizeof(mxfp8_gemm_desc)) == 0;
}

// One entry per device ordinal: the last request seen there and the Plan
// built for it.  get() works under the lock: make(Plan*) runs only when the
// device's last request differs (or none was seen), then refresh(Plan*) on
// every call (for per-call parts such as the activations' tensor map, which
// it may keep when they repeat too), then the plan is copied out.  A failed
// make or refresh leaves the entry empty.
template <class Plan, int kDevices>
class LastRequestCache {
 public:
  template <class Make, class Refresh>
  mxfp8_status get(int device, const NoallocRequest& request, Plan* out, Make make,
                   Refresh refresh) {
    if (device < 0 || device >= kDevices) return MXFP8_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(mutex_);
    Entry& e = entries_[device];
    if (!e.valid || !same_request(e.request, request)) {
      e.valid = false;
      e.plan = Plan{};
      const mxfp8_status st = make(&e.plan);
      if (st != MXFP8_OK) return st;
      e.request = request;
      e.valid = true;
    }
    const mxfp8_status st = refresh(&e.plan);
    if (st != MXFP8_OK) {
      e.valid = false;
      return st;
    }
    *out = e.plan;
    return MXFP8_OK;
  }

 private:
  struct Entry {
    bool valid = false;
    NoallocRequest request{};
    Plan plan{};
  };
  std::mutex mutex_;
  Entry entries_[kDevices];
};

}  // namespace mxfp8
