// Host-only check of the allocation-free call's set-up memo (compiled with
// g++ by tests/test_noalloc_cache_cpu.py; no CUDA runtime involved): a call
// that repeats the previous call's device, weight pointer and descriptor
// reuses the plan built for it, so the tensor map is not encoded again;
// anything else that differs builds a new plan; devices keep their own
// entries; a failed build leaves nothing behind.  Prints one line per check
// and exits non-zero on the first failure.
#include <cstdio>
#include <cstdlib>

#include "noalloc_cache.h"

namespace {

struct Plan {
  int built_for = -1;  // which make() call built it
  int refreshed = 0;   // how many refresh() calls it has seen
};

int makes = 0;

int check(bool ok, const char* what) {
  std::printf("%s %s\n", ok ? "ok" : "FAIL", what);
  if (!ok) std::exit(1);
  return 0;
}

mxfp8_gemm_desc desc_of(int n, int k, int split_k) {
  mxfp8_gemm_desc d{};
  d.n = n;
  d.k = k;
  d.capacity_m = 8;
  d.split_k = split_k;
  return d;
}

}  // namespace

int main() {
  mxfp8::LastRequestCache<Plan, 4> cache;
  auto make = [](Plan* p) {
    p->built_for = makes++;
    return MXFP8_OK;
  };
  auto refresh = [](Plan* p) {
    ++p->refreshed;
    return MXFP8_OK;
  };
  int w0 = 0, w1 = 0;
  const mxfp8::NoallocRequest a{&w0, desc_of(1024, 4096, 2)};
  Plan out;

  check(cache.get(0, a, &out, make, refresh) == MXFP8_OK && makes == 1 && out.built_for == 0,
        "first call builds the plan");
  check(cache.get(0, a, &out, make, refresh) == MXFP8_OK && makes == 1 && out.built_for == 0 &&
            out.refreshed == 2,
        "an identical second call reuses it (no second encode) and still refreshes");

  mxfp8::NoallocRequest b = a;
  b.w = &w1;
  check(cache.get(0, b, &out, make, refresh) == MXFP8_OK && makes == 2 && out.built_for == 1 &&
            out.refreshed == 1,
        "another weight pointer builds a new plan");

  mxfp8::NoallocRequest c = b;
  c.desc.stages = 6;
  check(cache.get(0, c, &out, make, refresh) == MXFP8_OK && makes == 3,
        "any other descriptor field builds a new plan");
  c.desc.wait_limit_ms = 10;
  check(cache.get(0, c, &out, make, refresh) == MXFP8_OK && makes == 4,
        "the last descriptor field counts too");

  check(cache.get(1, a, &out, make, refresh) == MXFP8_OK && makes == 5,
        "another device keeps its own entry");
  check(cache.get(0, c, &out, make, refresh) == MXFP8_OK && makes == 5,
        "and leaves the first device's entry in place");

  auto failing = [](Plan*) { return MXFP8_ERR_CUDA; };
  check(cache.get(2, a, &out, failing, refresh) == MXFP8_ERR_CUDA, "a failed build reports it");
  check(cache.get(2, a, &out, make, refresh) == MXFP8_OK && makes == 6,
        "and leaves no entry: the next call builds");

  auto bad_refresh = [](Plan*) { return MXFP8_ERR_CUDA; };
  check(cache.get(2, a, &out, make, bad_refresh) == MXFP8_ERR_CUDA && makes == 6,
        "a failed refresh reports it");
  check(cache.get(2, a, &out, make, refresh) == MXFP8_OK && makes == 7,
        "and drops the entry");

  check(cache.get(-1, a, &out, make, refresh) == MXFP8_ERR_UNSUPPORTED &&
            cache.get(4, a, &out, make, refresh) == MXFP8_ERR_UNSUPPORTED && makes == 7,
        "device ordinals outside the table are refused without a build");
  return 0;
}
