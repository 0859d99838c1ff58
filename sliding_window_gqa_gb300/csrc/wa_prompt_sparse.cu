// wa_prompt_sparse.cu — block-sparse prompt form: instantiations and launches.
//
// The kernel is in wa_prompt_kernel.cuh (the block-sparse form is described there).
#include "wa_prompt_kernel.cuh"

namespace wa {

cudaError_t prompt_sparse_prepare_device(int) {
    cudaError_t e;
    if ((e = get_encoder()) != cudaSuccess) return e;
    if ((e = set_attr<128, 1, true>()) != cudaSuccess) return e;
    if ((e = set_attr<128, 2, true>()) != cudaSuccess) return e;
    if ((e = set_attr<128, 3, true>()) != cudaSuccess) return e;
    if ((e = set_attr<256, 1, true>()) != cudaSuccess) return e;
    if ((e = set_attr<256, 2, true>()) != cudaSuccess) return e;
    return set_attr<256, 3, true>();
}

cudaError_t launch_prompt_sparse(const PromptArgs& a, cudaStream_t s) {
    if (get_encoder() != cudaSuccess) return cudaErrorNotSupported;
    if (a.d == 256) {
        if (a.p32 == 2) return launch_t<256, 3, true>(a, s);
        return a.p32 ? launch_t<256, 2, true>(a, s) : launch_t<256, 1, true>(a, s);
    }
    if (a.p32 == 2) return launch_t<128, 3, true>(a, s);
    return a.p32 ? launch_t<128, 2, true>(a, s) : launch_t<128, 1, true>(a, s);
}

}  // namespace wa
