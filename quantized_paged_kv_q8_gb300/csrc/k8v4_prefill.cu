// Chunked-prefill attention (tcgen05 tensor cores).  Placeholder until the
// tensor-core kernel lands: the call reports an invalid argument.
#include "k8v4_common.cuh"

namespace k8v4 {
int launch_prefill(const Launch&, const CacheView&, const void*, const int32_t*, int64_t, int, int,
                   const int32_t*, float, float*) {
  return K8V4_EINVAL;
}
}  // namespace k8v4
