// Packed causal prefill (placeholder until the tensor-core kernel lands).
#include "pkv_internal.h"

cudaError_t launch_prefill(pkv_cache *, const PrefillLaunch &, cudaStream_t) { return cudaErrorNotSupported; }
