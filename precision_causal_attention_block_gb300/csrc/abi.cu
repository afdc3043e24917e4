// Library-wide pieces of the C ABI: status strings and the driver entry
// point for tensor-map encoding (resolved at run time, so loading the
// library needs no libcuda at link time).
#include <atomic>
#include <mutex>

#include "common.cuh"

namespace flamia {

EncodeTiledFn get_encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

namespace {
std::atomic<unsigned long long> g_launches{0};
}

void count_launches(int n) { g_launches.fetch_add(static_cast<unsigned long long>(n)); }

}  // namespace flamia

extern "C" unsigned long long flamia_debug_launch_count(void) { return flamia::g_launches.load(); }

extern "C" const char* flamia_status_str(flamia_status s) {
  switch (s) {
    case FLAMIA_OK: return "ok";
    case FLAMIA_ERR_INVALID_ARG: return "invalid argument";
    case FLAMIA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FLAMIA_ERR_WORKSPACE: return "workspace or work-list buffer too small";
    case FLAMIA_ERR_CUDA: return "CUDA runtime error";
  }
  return "unknown status";
}
