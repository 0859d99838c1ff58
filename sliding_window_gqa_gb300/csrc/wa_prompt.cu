// wa_prompt.cu — prompt form (placeholder until the tensor-core kernel lands).
#include "wa_internal.h"

namespace wa {

cudaError_t prompt_prepare_device(int) { return cudaSuccess; }

cudaError_t launch_prompt(const PromptArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace wa
