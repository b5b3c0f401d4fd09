// Decode kernels for model dtype PKV_F16 with KV dtype PKV_F16 (one translation unit per pair so
// that the instantiations compile in parallel).
#include "decode_impl.cuh"

cudaError_t pkv_decode_f16(const pkv_decode::Args &a, int D, int G, int grid, size_t smem, cudaStream_t st,
                          bool merge) {
    return pkv_decode::dispatch<PKV_F16, PKV_F16>(a, D, G, grid, smem, st, merge);
}

int pkv_decode_occupancy_f16(int D, int G, size_t smem) { return pkv_decode::occupancy_dispatch<PKV_F16, PKV_F16>(D, G, smem); }
