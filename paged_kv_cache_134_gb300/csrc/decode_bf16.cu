// Decode kernels for model dtype PKV_BF16 with KV dtype PKV_BF16 (one translation unit per pair so
// that the instantiations compile in parallel).
#include "decode_impl.cuh"

cudaError_t pkv_decode_bf16(const pkv_decode::Args &a, int D, int G, int grid, size_t smem, cudaStream_t st,
                          bool merge) {
    return pkv_decode::dispatch<PKV_BF16, PKV_BF16>(a, D, G, grid, smem, st, merge);
}

int pkv_decode_occupancy_bf16(int D, int G, size_t smem) { return pkv_decode::occupancy_dispatch<PKV_BF16, PKV_BF16>(D, G, smem); }
