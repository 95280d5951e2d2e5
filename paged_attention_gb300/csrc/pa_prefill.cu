// pa_prefill.cu -- tcgen05 prefill (placeholder until the kernel lands).
#include "pa_internal.cuh"

namespace pa {

int prefill_smem_bytes(int, bool) { return -1; }
const void* prefill_kernel_ptr(int, bool) { return nullptr; }
cudaError_t launch_prefill_from_api(const pa_problem&, const WsLayout&, const void*,
                                    const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,
                                    const int32_t*, const int32_t*, const int32_t*, const float*,
                                    const float*, void*, void*, void*, float*, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace pa
