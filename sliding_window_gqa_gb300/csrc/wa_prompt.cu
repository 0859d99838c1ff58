// wa_prompt.cu — prompt form (dense rows): instantiations, the tensor-map encoder, launches.
//
// The kernels are in wa_prompt_d256.cuh (head dim 256 with one or two P parts),
// wa_prompt_pair.cuh (head dim 128 with one or two P parts) and wa_prompt_kernel.cuh (three P
// parts at either head dim); see there for the designs and sources.
#include <mutex>

#include "wa_prompt_kernel.cuh"
#include "wa_prompt_pair.cuh"
#include "wa_prompt_d256.cuh"

namespace wa {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn_ptr = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn_ptr = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return fn_ptr;
}

cudaError_t prompt_prepare_device(int) {
    cudaError_t e;
    if ((e = get_encoder()) != cudaSuccess) return e;
    if ((e = set_pair_attr<1>()) != cudaSuccess) return e;
    if ((e = set_pair_attr<2>()) != cudaSuccess) return e;
    if ((e = set_attr<128, 3>()) != cudaSuccess) return e;
    if ((e = set_d256_attr<1>()) != cudaSuccess) return e;
    if ((e = set_d256_attr<2>()) != cudaSuccess) return e;
    return set_attr<256, 3>();
}

cudaError_t launch_prompt(const PromptArgs& a, cudaStream_t s) {
    if (get_encoder() != cudaSuccess) return cudaErrorNotSupported;
    if (a.d == 256) {
        if (a.p32 == 2) return launch_t<256, 3, false>(a, s);
        return a.p32 ? launch_d256<2>(a, s) : launch_d256<1>(a, s);
    }
    if (a.p32 == 2) return launch_t<128, 3, false>(a, s);
    return a.p32 ? launch_pair<2>(a, s) : launch_pair<1>(a, s);
}

}  // namespace wa
