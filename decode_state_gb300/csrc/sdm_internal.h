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
    // the inputs' row of (token t, stream s) is t * tstride + s * sstride, and so is the readings'
    // row: time-major [T, S, .] has (S, 1), the stream-major layout [S, T, .] has (1, T)
    int64_t tstride, sstride;
    int slice_cols;   // columns one block owns (the last slice may be narrower)
    int n_slices;     // ceil(hd / slice_cols)
    int stream_rows;    // rows per ring chunk of the streaming path
    int stream_stages;  // chunk buffers in its ring (3 or 4)
    int piece_write;  // staged path: decay-and-write by 16-byte pieces where they tile the threads
    int inputs_ready; // the inputs predate the preceding kernel: load them before waiting on it
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
    void* stash;             // [tokens, width[0], hd], or the compact snapshot when kpos is set
    const int32_t* kpos;     // [tokens, width[0]] compact-snapshot rows (-1: none), or nullptr
    int64_t tokens;
    int chunk, valid;
    const int32_t* chunk_valid;
    int slice_cols, n_slices;
    int inputs_ready;  // the index and weight rows predate the preceding kernel: load them before waiting
};

// A resolved gather launch: the kernel instance, its geometry and every kernel argument.
struct GatherLaunch {
    const void* fn;  // kernel (host stub of the template instance); nullptr: nothing to launch
    GatherArgs a;
    int stash_bulk, early_trigger;
    unsigned int grid, block;
    size_t smem;
};

// A resolved decode launch: the kernel instance, its geometry and every kernel argument.
struct DecodeLaunch {
    const void* fn;  // kernel (host stub of the template instance); nullptr: nothing to launch
    DecodeArgs a;
    int early_trigger;
    unsigned int grid, block;
    size_t smem;
};

// Validated launches (arguments already checked by the ABI layer). Return a cudaError_t.
int launch_decode(const DecodeArgs& a, int bank_dtype, int idx_dtype, cudaStream_t stream);
// launch_decode in two halves: choose the kernel and geometry (device queries, no launch), then launch.
int plan_decode(const DecodeArgs& a, int bank_dtype, int idx_dtype, DecodeLaunch* L);
int run_decode(const DecodeLaunch& L, cudaStream_t stream);
int launch_gather(const GatherArgs& a, int bank_dtype, int idx_dtype, int w_dtype, cudaStream_t stream);
// launch_gather in two halves: choose the kernel and geometry (device queries, no launch), then launch.
int plan_gather(const GatherArgs& a, int bank_dtype, int idx_dtype, int w_dtype, GatherLaunch* L);
int run_gather(const GatherLaunch& L, cudaStream_t stream);

// Device status words of the kernel files (OR of SDM_DEV_* bits); read and optionally reset.
int decode_status(unsigned int* word, bool clear);
int gather_status(unsigned int* word, bool clear);

// Multiprocessor count of the current device (cached per device).
int sm_count();
// Shared memory of one multiprocessor, and the part the system reserves per block, in bytes
// (current device, cached per device).
size_t smem_per_sm();
size_t smem_reserved_per_block();

// Let `kernel` use `smem` bytes of dynamic shared memory (raises the limit above the default 48 KB
// on the current device). Called before any occupancy query of that launch, so that the query sees
// the launch's real limit. The limit only ever grows (to the largest size asked for so far per
// kernel and device), so that concurrent callers cannot lower it under each other, and a kernel
// whose limit already suffices costs no runtime call. Returns a cudaError_t.
int allow_smem(const void* kernel, size_t smem);

// Blocks of `kernel` resident per SM with `threads` threads and `smem` bytes of dynamic shared
// memory on the current device (0 when the query fails), cached per host thread.
int blocks_per_sm(const void* kernel, int threads, size_t smem);

// Launch the kernel at address `kernel` (arguments as an array of pointers to them) with
// programmatic stream serialization (see grid_dependency_wait). The dynamic shared-memory limit
// must already allow `smem` (allow_smem). Returns the cudaError_t of the launch call itself; the
// error state of the runtime is consumed only when that call failed, so an earlier error left by
// other code is neither reported nor cleared here.
inline int launch_pdl_raw(const void* kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, void** args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelExC(&cfg, kernel, args);
    if (e != cudaSuccess) (void)cudaGetLastError();
    return (int)e;
}

}  // namespace sdm
