// Internal interface between the C-ABI layer (sdm_abi.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sdm {

// Launch arguments of the decode kernels (single token: T == 1).
struct DecodeArgs {
    void* bank;
    const void* k_idx;
    const float* k_val;
    const float* v;
    const float* beta;
    const float* g;
    const void* q_idx;
    const float* q_val;
    void* out;
    int64_t n_streams;
    int hd, W, R, G, T;
    int slice_cols;  // columns one block owns (the last slice may be narrower)
    int n_slices;    // ceil(hd / slice_cols)
};

struct GatherArgs {
    const void* bank;
    int64_t n_slots;
    int hd;
    int n_ops;
    const void* idx[2];
    const void* w[2];
    float* out[2];
    int width[2];
    void* stash;
    int64_t tokens;
    int chunk, valid;
    const int32_t* chunk_valid;
    int slice_cols, n_slices;
};

// Validated launches (arguments already checked by the ABI layer). Return a cudaError_t.
int launch_decode(const DecodeArgs& a, int bank_dtype, int idx_dtype, cudaStream_t stream);
int launch_gather(const GatherArgs& a, int bank_dtype, int idx_dtype, int w_dtype, cudaStream_t stream);

// Device status words of the kernel files (OR of SDM_DEV_* bits); read and optionally reset.
int decode_status(unsigned int* word, bool clear);
int gather_status(unsigned int* word, bool clear);

// Multiprocessor count of the current device (cached per device).
int sm_count();

}  // namespace sdm
