// SDM decode: one write-then-read token per stream (T == 1), or T tokens per stream in one
// persistent launch.
//
// Math (sparse-delta-memory 2.0.0, decode.py, sdm_decode_step docstring): per stream, with
// d = exp(g),
//     retrieved   = sum_w k_val[w] * d[w] * bank[k_idx[w]]
//     delta_v     = beta * (v - retrieved)
//     bank[k_w]   = d[w] * bank[k_w] + k_val[w] * delta_v
//     readings    = sum_r q_val[r] * bank[q_idx[r]]         (after the write)
// k_val, v and q_val rounded to the bank dtype; beta and g in float32; readings in the bank dtype.
//
// Design. One block owns one (stream, column slice) for every token it runs, so it is the only
// writer and reader of those columns of the stream's private slots; a block barrier therefore
// orders a token's writes before its reads and before the next token's retrieve (the argument
// the reference kernel makes for its CTA barrier). Per token:
//   1. the slots, rounded weights and gates go to shared memory;
//   2. warp 0 issues one bulk copy (cp.async.bulk, async proxy) per write row slice into shared
//      memory, all W in flight at once, completion counted on an mbarrier;
//   3. each thread owns CPT adjacent columns and runs the retrieve as one fmaf chain over
//      ascending w, then delta, then the decay-and-write, storing the new row slices to global
//      memory with plain stores;
//   4. fence.proxy.async.global + barrier make those stores visible to the next bulk copies;
//   5. warp 0 bulk-copies the R read rows, each thread reduces its columns over ascending r and
//      stores the readings.
// Rows whose length is not a multiple of 16 bytes (or an unaligned bank) take a plain-load path
// with one column per thread; a thread then only ever touches its own column, so program order
// alone orders its writes and reads.
//
// Arithmetic per element (float32, no other fusion):
//   a_w = kv_w * d_w;  retrieved = fmaf(a_w, row_w, .) over w;  delta = beta * (round(v) - retrieved)
//   new_w = fmaf(kv_w, delta, row_w * d_w);  readings = fmaf(qv_r, row_r, .) over r
// with d_w the float32 nearest to e^g (computed in double precision and rounded once).
#include <algorithm>
#include <climits>

#include "../../include/sdm.h"
#include "sdm_device.cuh"
#include "sdm_internal.h"

namespace sdm {
namespace {

__device__ unsigned int g_decode_status;

constexpr int kMaxThreads = 256;
constexpr size_t kRowsBudget = 32 * 1024;  // staged rows of one block; with the metadata this stays under 48 KB

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Shared-memory layout of one block (host and device agree on it).
struct SmemLayout {
    size_t rows, k_slot, q_slot, kv, aw, dw, qv, bar, total;
    __host__ __device__ SmemLayout(int W, int R, int slice_cols, int es) {
        const int maxwr = W > R ? W : R;
        rows = 0;
        k_slot = align_up((size_t)maxwr * slice_cols * es, 16);
        q_slot = k_slot + (size_t)W * 8;
        kv = q_slot + (size_t)R * 8;
        aw = kv + (size_t)W * 4;
        dw = aw + (size_t)W * 4;
        qv = dw + (size_t)W * 4;
        bar = align_up(qv + (size_t)R * 4, 8);
        total = bar + 8;
    }
};

// Warp 0: bulk-copy n row slices (row_bytes each, starting at column c0) into rows[i * sw].
template <typename E>
__device__ __forceinline__ void issue_rows(E* rows, const E* bank, const int64_t* slot, int n, int hd, int c0,
                                           int sw, uint32_t row_bytes, uint64_t* bar) {
    const int lane = threadIdx.x;
    if (lane == 0) mbar_arrive_expect_tx(bar, row_bytes * (uint32_t)n);
    __syncwarp();
    for (int i = lane; i < n; i += 32) bulk_g2s(rows + (size_t)i * sw, bank + slot[i] * hd + c0, row_bytes, bar);
}

// Plain-load path: this thread's column of n rows into rows[i * sw + j].
template <typename E>
__device__ __forceinline__ void load_rows_simt(E* rows, const E* bank, const int64_t* slot, int n, int hd, int col,
                                               int sw, int j) {
    int i = 0;
    for (; i + 8 <= n; i += 8) {
        E x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) x[u] = bank[slot[i + u] * hd + col];
#pragma unroll
        for (int u = 0; u < 8; ++u) rows[(size_t)(i + u) * sw + j] = x[u];
    }
    for (; i < n; ++i) rows[(size_t)i * sw + j] = bank[slot[i] * hd + col];
}

// CPT adjacent elements of a staged row, widened to float32.
template <typename E, int CPT>
__device__ __forceinline__ void read_staged(const E* p, float (&x)[CPT]) {
    if constexpr (CPT == 2) {
        const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
        x[0] = __uint_as_float(u << 16);
        x[1] = __uint_as_float(u & 0xffff0000u);
    } else {
        x[0] = to_f32(p[0]);
    }
}

template <typename E, int CPT>
__device__ __forceinline__ void store_elems(E* p, const float (&x)[CPT]) {
    if constexpr (CPT == 2) {
        *reinterpret_cast<uint32_t*>(p) = pack_bf16x2(x[0], x[1]);
    } else {
        p[0] = from_f32<E>(x[0]);
    }
}

// Wait for the current bulk phase; on a timeout every thread of the block learns it at the
// barrier, the block records SDM_DEV_TIMEOUT, waits once more (bounded) for its copies and
// reports that it must stop.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t& parity, int* s_abort) {
    const bool ok = mbar_wait_bounded(bar, parity, kWaitLimitNs);
    if (!ok) atomicOr(s_abort, 1);
    __syncthreads();
    if (*s_abort) {
        if (threadIdx.x == 0) atomicOr(&g_decode_status, SDM_DEV_TIMEOUT);
        if (!ok) mbar_wait_bounded(bar, parity, kWaitLimitNs);
        return false;
    }
    parity ^= 1u;
    return true;
}

template <typename E, typename I, bool BULK>
__global__ void __launch_bounds__(kMaxThreads) decode_kernel(const DecodeArgs a) {
    constexpr int ES = sizeof(E);
    constexpr int CPT = (BULK && ES == 2) ? 2 : 1;
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_abort;

    const int W = a.W, R = a.R, G = a.G, hd = a.hd, sw = a.slice_cols;
    const SmemLayout L(W, R, sw, ES);
    E* rows = reinterpret_cast<E*>(smem + L.rows);
    int64_t* k_slot = reinterpret_cast<int64_t*>(smem + L.k_slot);
    int64_t* q_slot = reinterpret_cast<int64_t*>(smem + L.q_slot);
    float* kv = reinterpret_cast<float*>(smem + L.kv);
    float* aw = reinterpret_cast<float*>(smem + L.aw);
    float* dw = reinterpret_cast<float*>(smem + L.dw);
    float* qv = reinterpret_cast<float*>(smem + L.qv);
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + L.bar);

    const int tid = threadIdx.x, nt = blockDim.x;
    const int64_t s = blockIdx.x / a.n_slices;
    const int c0 = (int)(blockIdx.x % a.n_slices) * sw;
    const int ncols = min(sw, hd - c0);
    const int j = tid * CPT;  // this thread's first column within the slice
    const bool active = j < ncols;
    const uint32_t row_bytes = (uint32_t)ncols * ES;
    E* bank = static_cast<E*>(a.bank);
    E* out = static_cast<E*>(a.out);

    if (tid == 0) {
        s_abort = 0;
        if (BULK) {
            mbar_init(bar, 1);
            mbar_init_fence();
        }
    }
    __syncthreads();
    uint32_t parity = 0;

    for (int t = 0; t < a.T; ++t) {
        const int64_t ts = (int64_t)t * a.n_streams + s;  // (token, stream) row of the time-major inputs

        // 1. per-token metadata
        for (int i = tid; i < W; i += nt) {
            const int64_t e = ts * W + i;
            k_slot[i] = load_index<I>(a.k_idx, e);
            kv[i] = round_to<E>(__ldg(a.k_val + e));
            if (G != 1) dw[i] = (float)exp((double)__ldg(a.g + ts * G + i));
        }
        if (G == 1 && tid == 0) dw[0] = (float)exp((double)__ldg(a.g + ts));
        for (int i = tid; i < R; i += nt) {
            const int64_t e = ts * R + i;
            q_slot[i] = load_index<I>(a.q_idx, e);
            qv[i] = round_to<E>(__ldg(a.q_val + e));
        }
        float vr[CPT];
#pragma unroll
        for (int k = 0; k < CPT; ++k) vr[k] = active ? round_to<E>(__ldg(a.v + ts * hd + c0 + j + k)) : 0.0f;
        const float beta = __ldg(a.beta + ts);
        __syncthreads();

        // 2. the write rows
        if (BULK) {
            if (tid < 32) issue_rows<E>(rows, bank, k_slot, W, hd, c0, sw, row_bytes, bar);
        } else if (active) {
            load_rows_simt<E>(rows, bank, k_slot, W, hd, c0 + j, sw, j);
        }
        for (int i = tid; i < W; i += nt) aw[i] = __fmul_rn(kv[i], dw[G == 1 ? 0 : i]);
        if (BULK) {
            if (!wait_phase(bar, parity, &s_abort)) return;
        } else {
            __syncthreads();
        }

        // 3. retrieve, delta, decay-and-write for this thread's columns
        if (active) {
            float acc[CPT];
#pragma unroll
            for (int k = 0; k < CPT; ++k) acc[k] = 0.0f;
            for (int w = 0; w < W; ++w) {
                float x[CPT];
                read_staged<E, CPT>(rows + (size_t)w * sw + j, x);
                const float a_w = aw[w];
#pragma unroll
                for (int k = 0; k < CPT; ++k) acc[k] = fmaf(a_w, x[k], acc[k]);
            }
            float delta[CPT];
#pragma unroll
            for (int k = 0; k < CPT; ++k) delta[k] = __fmul_rn(beta, __fsub_rn(vr[k], acc[k]));
            for (int w = 0; w < W; ++w) {
                float x[CPT], y[CPT];
                read_staged<E, CPT>(rows + (size_t)w * sw + j, x);
                const float kvw = kv[w], dww = dw[G == 1 ? 0 : w];
#pragma unroll
                for (int k = 0; k < CPT; ++k) y[k] = fmaf(kvw, delta[k], __fmul_rn(x[k], dww));
                store_elems<E, CPT>(bank + k_slot[w] * hd + c0 + j, y);
            }
        }
        if (BULK) fence_proxy_async_global();
        __syncthreads();

        // 4. the read rows, after the write
        if (BULK) {
            if (tid < 32) issue_rows<E>(rows, bank, q_slot, R, hd, c0, sw, row_bytes, bar);
            if (!wait_phase(bar, parity, &s_abort)) return;
        } else if (active) {
            load_rows_simt<E>(rows, bank, q_slot, R, hd, c0 + j, sw, j);
        }

        // 5. readings
        if (active) {
            float acc[CPT];
#pragma unroll
            for (int k = 0; k < CPT; ++k) acc[k] = 0.0f;
            for (int r = 0; r < R; ++r) {
                float x[CPT];
                read_staged<E, CPT>(rows + (size_t)r * sw + j, x);
                const float q = qv[r];
#pragma unroll
                for (int k = 0; k < CPT; ++k) acc[k] = fmaf(q, x[k], acc[k]);
            }
            store_elems<E, CPT>(out + ts * hd + c0 + j, acc);
        }
        __syncthreads();  // metadata and rows are rewritten by the next token
    }
}

template <typename E, typename I, bool BULK>
int launch_typed(const DecodeArgs& a, dim3 grid, dim3 block, size_t smem, cudaStream_t stream) {
    decode_kernel<E, I, BULK><<<grid, block, smem, stream>>>(a);
    return (int)cudaGetLastError();
}

template <typename E, typename I>
int launch_bulk_or_simt(bool bulk, const DecodeArgs& a, dim3 grid, dim3 block, size_t smem, cudaStream_t stream) {
    return bulk ? launch_typed<E, I, true>(a, grid, block, smem, stream)
                : launch_typed<E, I, false>(a, grid, block, smem, stream);
}

int shrink_cols(int sw, bool bulk, int es) {
    const int q = bulk ? 16 / es : 32;
    const int half = (sw / 2 + q - 1) / q * q;
    return std::max(q, half);
}

}  // namespace

int launch_decode(const DecodeArgs& a0, int bank_dtype, int idx_dtype, cudaStream_t stream) {
    DecodeArgs a = a0;
    if (a.n_streams == 0 || a.T == 0) return 0;
    const int es = bank_dtype == SDM_BF16 ? 2 : 4;
    const bool bulk = ((int64_t)a.hd * es) % 16 == 0 && reinterpret_cast<uintptr_t>(a.bank) % 16 == 0;
    const int cpt = (bulk && es == 2) ? 2 : 1;
    const int maxwr = std::max(a.W, a.R);

    // Column slice: the whole row when it fits; narrower to bound shared memory and to give the
    // grid at least two blocks per SM when there are few streams.
    int sw = std::min(a.hd, kMaxThreads * cpt);
    if (bulk) sw = sw / (16 / es) * (16 / es);
    while ((size_t)maxwr * sw * es > kRowsBudget && sw > (bulk ? 16 / es : 32)) sw = shrink_cols(sw, bulk, es);
    const int64_t want_blocks = 2LL * sm_count();
    while (a.n_streams * ((a.hd + sw - 1) / sw) < want_blocks && sw * es > 128) {
        const int next = shrink_cols(sw, bulk, es);
        if (next >= sw) break;
        sw = next;
    }
    a.slice_cols = sw;
    a.n_slices = (a.hd + sw - 1) / sw;
    const int64_t blocks = a.n_streams * a.n_slices;
    if (blocks > INT_MAX) return SDM_ECOUNT;
    const int threads = ((sw + cpt - 1) / cpt + 31) / 32 * 32;
    const size_t smem = SmemLayout(a.W, a.R, sw, es).total;

    const dim3 grid((unsigned)blocks), block((unsigned)threads);
    if (bank_dtype == SDM_BF16) {
        return idx_dtype == SDM_I32 ? launch_bulk_or_simt<uint16_t, int32_t>(bulk, a, grid, block, smem, stream)
                                    : launch_bulk_or_simt<uint16_t, int64_t>(bulk, a, grid, block, smem, stream);
    }
    return idx_dtype == SDM_I32 ? launch_bulk_or_simt<float, int32_t>(bulk, a, grid, block, smem, stream)
                                : launch_bulk_or_simt<float, int64_t>(bulk, a, grid, block, smem, stream);
}

int decode_status(unsigned int* word, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(word, g_decode_status, sizeof(unsigned int));
    if (e == cudaSuccess && clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_decode_status, &zero, sizeof(unsigned int));
    }
    return (int)e;
}

}  // namespace sdm
