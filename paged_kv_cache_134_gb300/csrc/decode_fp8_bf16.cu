// Decode kernels for model dtype PKV_BF16 with KV dtype PKV_FP8_E4M3 (one translation unit per pair so
// that the instantiations compile in parallel).
#include "decode_impl.cuh"

cudaError_t pkv_decode_fp8_bf16(const pkv_decode::Args &a, int D, int G, int grid, int threads, size_t smem,
                          cudaStream_t st, int *occ) {
    return pkv_decode::dispatch<PKV_BF16, PKV_FP8_E4M3>(a, D, G, grid, threads, smem, st, occ);
}
