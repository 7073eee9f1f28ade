// SDM token gather.
//
// Math (sparse-delta-memory 2.0.0, cuda/gather_cuda.py, module docstring): for every token t and
// operand o,
//     out_o[t]    = sum_n w_o[t, n] * bank[idx_o[t, n]]     (float32 accumulation)
//     stash[t, n] = bank[idx_0[t, n]]                       (raw rows of operand 0)
// and a token whose position in its chunk is >= valid is padding: it reads nothing and gets zero
// outputs and zero stash rows.
//
// Design. One block owns one (token, column slice, operand): two small blocks per token rather
// than one block over both operands keep twice the independent chains (index load, then rows)
// resident per SM in the same shared memory. Every thread issues 16-byte cp.async copies of the
// operand's entry row slices (all in flight at once) into shared memory; the stash
// rows then leave shared memory by bulk stores (one cp.async.bulk store for the whole token when
// the slice is the full row, its lines marked evict-first in L2: the kernel never reads them),
// while each column is reduced over the entries in ascending order with fmaf (the reference's
// order with one row group). The block has a thread per column of the slice, all of which copy
// rows: whole blocks of column pairs (half the threads) measured 6 % slower. The reduction itself
// runs one column per thread, except for bf16 rows and weights in the full 128-column slice, where
// the first half of the threads each sum a column pair (fewer loads and unpackings per column). The
// row loads use 16-byte copies rather than one bulk copy per row: with 256-byte rows the bulk-copy
// engine sustained about 3 TB/s of row reads per GPU. Rows that are not a multiple of 16 bytes, or
// an unaligned bank, take a plain-load path with one column per thread. Row indices outside
// [0, n_slots) are skipped (zero row) and flagged in the status word.
//
// Compact-snapshot form (kpos set): instead of the stash, operand 0's row of entry n goes to row
// kpos[t, n] of the chunk's block of chunk * W0 rows when kpos >= 0; each thread stores the 16-byte
// pieces it copied itself as soon as they have landed, so the form costs no extra barrier.
#include <algorithm>
#include <climits>

#include "sdm.h"
#include "sdm_device.cuh"
#include "sdm_internal.h"

namespace sdm {
namespace {

__device__ unsigned int g_gather_status;

constexpr int kMaxThreads = 256;
constexpr size_t kRowsBudget = 40 * 1024;
constexpr int kFullSlice = 128;  // the slice width with its own kernel instance

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct GatherLayout {
    size_t rows, slot, wt, kp, total;
    __host__ __device__ GatherLayout(int n_rows, int slice_cols, int es) {
        rows = 0;
        slot = align_up((size_t)n_rows * slice_cols * es, 16);
        wt = align_up(slot + (size_t)n_rows * 8, 16);  // float weights, or raw bf16 ones
        kp = align_up(wt + (size_t)n_rows * 4, 16);    // compact-snapshot rows of operand 0's entries
        total = kp + (size_t)n_rows * 4;
    }
};

// bf16 weights over a bf16 bank stay raw: both operands of the mixed-precision fma below
template <typename E, typename WT>
constexpr bool kRawWeights = sizeof(E) == 2 && sizeof(WT) == 2;

// acc + w * x for bf16 w and x: the product of two bf16 values is exact in float32, so this single
// rounding gives the same float32 as widening both and calling fmaf
__device__ __forceinline__ float fma_bf16(uint16_t w, uint16_t x, float acc) {
    asm("fma.rn.f32.bf16 %0, %1, %2, %0;" : "+f"(acc) : "h"(w), "h"(x));
    return acc;
}

// one column's weighted sum over the NR staged rows (x: the column's element of row 0, rows sw
// elements apart), one chain over ascending entries
template <typename E, typename WT>
__device__ __forceinline__ float weighted_sum(const E* x, int sw, const unsigned char* wts, int NR) {
    float acc = 0.0f;
    int n = 0;
    if constexpr (kRawWeights<E, WT>) {
        const uint16_t* w = reinterpret_cast<const uint16_t*>(wts);
        for (; n + 8 <= NR; n += 8) {
            const uint4 w8 = *reinterpret_cast<const uint4*>(w + n);
            const uint32_t wp[4] = {w8.x, w8.y, w8.z, w8.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                acc = fma_bf16((uint16_t)(wp[u] & 0xffffu), x[(size_t)(n + 2 * u) * sw], acc);
                acc = fma_bf16((uint16_t)(wp[u] >> 16), x[(size_t)(n + 2 * u + 1) * sw], acc);
            }
        }
        for (; n < NR; ++n) acc = fma_bf16(w[n], x[(size_t)n * sw], acc);
    } else {
        const float* w = reinterpret_cast<const float*>(wts);
        for (; n + 4 <= NR; n += 4) {
            const float4 w4 = *reinterpret_cast<const float4*>(w + n);
            acc = fmaf(w4.x, to_f32(x[(size_t)(n + 0) * sw]), acc);
            acc = fmaf(w4.y, to_f32(x[(size_t)(n + 1) * sw]), acc);
            acc = fmaf(w4.z, to_f32(x[(size_t)(n + 2) * sw]), acc);
            acc = fmaf(w4.w, to_f32(x[(size_t)(n + 3) * sw]), acc);
        }
        for (; n < NR; ++n) acc = fmaf(w[n], to_f32(x[(size_t)n * sw]), acc);
    }
    return acc;
}

// The weighted sums of two adjacent columns of bf16 rows with bf16 weights (x: the pair's elements
// of row 0, rows SW elements apart): one 32-bit load per row feeds both chains, so a thread does half
// the shared-memory loads and weight unpacking per column; each chain runs over ascending entries.
template <int SW>
__device__ __forceinline__ float2 weighted_sum_pair_bf16(const uint16_t* x, const unsigned char* wts, int NR) {
    const uint16_t* w = reinterpret_cast<const uint16_t*>(wts);
    float a0 = 0.0f, a1 = 0.0f;
    const auto row = [&](int n, uint16_t wv) {
        const uint32_t xv = *reinterpret_cast<const uint32_t*>(x + (size_t)n * SW);
        a0 = fma_bf16(wv, (uint16_t)(xv & 0xffffu), a0);
        a1 = fma_bf16(wv, (uint16_t)(xv >> 16), a1);
    };
    int n = 0;
    for (; n + 8 <= NR; n += 8) {
        const uint4 w8 = *reinterpret_cast<const uint4*>(w + n);
        const uint32_t wp[4] = {w8.x, w8.y, w8.z, w8.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            row(n + 2 * u, (uint16_t)(wp[u] & 0xffffu));
            row(n + 2 * u + 1, (uint16_t)(wp[u] >> 16));
        }
    }
    for (; n < NR; ++n) row(n, w[n]);
    return make_float2(a0, a1);
}

// Zero this block's slice of operand op's output, and for operand 0 its stash rows, of padding
// token t.
template <typename E>
__device__ void write_padding(const GatherArgs& a, int64_t t, int op, int c0, int j, bool active, bool flat16) {
    const int hd = a.hd, W0 = a.width[0];
    if (active) a.out[op][t * hd + c0 + j] = 0.0f;
    if (op != 0 || a.stash == nullptr || a.kpos != nullptr) return;  // the compact snapshot takes nothing from padding
    E* st = static_cast<E*>(a.stash) + t * W0 * hd;
    if (flat16) {  // the token's whole stash block is contiguous and 16-byte aligned
        uint4* p = reinterpret_cast<uint4*>(st);
        const int n16 = (int)((size_t)W0 * hd * sizeof(E) / 16);
        for (int i = threadIdx.x; i < n16; i += blockDim.x) p[i] = make_uint4(0u, 0u, 0u, 0u);
    } else if (active) {
        for (int n = 0; n < W0; ++n) st[(int64_t)n * hd + c0 + j] = E(0);
    }
}

// SW: the slice width in columns when it is known at compile time (the common full row of 128
// columns: row addresses in shared memory become immediate offsets), 0 when it is taken from the
// arguments.
template <typename E, typename I, typename WT, bool BULK, int SW>
__global__ void __launch_bounds__(kMaxThreads) gather_kernel(const GatherArgs a, int stash_bulk, int early_trigger) {
    constexpr int ES = sizeof(E);
    extern __shared__ __align__(128) unsigned char smem[];

    const int hd = a.hd, sw = SW ? SW : a.slice_cols;
    const int W0 = a.width[0], W1 = a.n_ops == 2 ? a.width[1] : 0;
    // one block per (token, column slice, operand): operand op's NR entries
    const int op = (int)(blockIdx.x % a.n_ops);
    const unsigned bx = blockIdx.x / a.n_ops;
    const int NR = op ? W1 : W0;
    const GatherLayout L(max(W0, W1), sw, ES);
    E* rows = reinterpret_cast<E*>(smem + L.rows);
    int64_t* slot = reinterpret_cast<int64_t*>(smem + L.slot);
    unsigned char* wt = smem + L.wt;
    int* kp = reinterpret_cast<int*>(smem + L.kp);

    const int tid = threadIdx.x, nt = blockDim.x;
    const int64_t t = bx / a.n_slices;
    const int c0 = (int)(bx % a.n_slices) * sw;
    const int ncols = min(sw, hd - c0);
    const int j = tid;  // this thread's column within the slice
    const bool active = j < ncols;
    const uint32_t row_bytes = (uint32_t)ncols * ES;
    const E* bank = static_cast<const E*>(a.bank);
    E* stash = static_cast<E*>(a.stash);

    // With inputs_ready the index and weight rows predate the preceding kernel: they are read, and
    // the rows they name warmed in L2, before waiting for that kernel; the bank is read and the
    // outputs written only after the wait (L2 is the point of coherence: a line warmed early still
    // holds every later write to it). The next launch is released only after the wait: released
    // at the start, whole chains of launches would sit waiting with their rows warmed far ahead
    // (a walk of plan slabs from a graph measured 6.1 instead of 3.9 us per launch).
    if (!a.inputs_ready) {
        grid_dependency_wait();
        if (early_trigger) grid_launch_dependents();
    }
    const int vt = a.chunk_valid != nullptr ? __ldg(a.chunk_valid + t / a.chunk) : a.valid;
    if ((int)(t % a.chunk) >= vt) {
        if (a.inputs_ready) {
            grid_dependency_wait();
            if (early_trigger) grid_launch_dependents();
        }
        write_padding<E>(a, t, op, c0, j, active, stash_bulk && a.n_slices == 1);
        return;
    }

    // this operand's entries
    for (int e = tid; e < NR; e += nt) {
        const int64_t i = t * NR + e;
        int64_t sl = load_index<I>(a.idx[op], i);
        if (sl < 0 || sl >= a.n_slots) {
            atomicOr(&g_gather_status, SDM_DEV_BAD_INDEX);
            sl = -1;
        }
        slot[e] = sl;
        if constexpr (kRawWeights<E, WT>)
            reinterpret_cast<uint16_t*>(wt)[e] = __ldg(static_cast<const uint16_t*>(a.w[op]) + i);
        else
            reinterpret_cast<float*>(wt)[e] = to_f32(__ldg(static_cast<const WT*>(a.w[op]) + i));
        if (a.kpos != nullptr && op == 0) {
            int k = __ldg(a.kpos + i);
            if (k >= a.chunk * W0 || (k >= 0 && sl < 0)) {
                if (k >= a.chunk * W0) atomicOr(&g_gather_status, SDM_DEV_BAD_INDEX);
                k = -1;
            }
            kp[e] = k;
        }
    }
    // compact snapshot: this token's chunk block
    E* compact = a.kpos != nullptr && op == 0 ? stash + (t / a.chunk) * ((int64_t)a.chunk * W0) * hd : nullptr;
    const bool stash_rows = stash != nullptr && a.kpos == nullptr && op == 0;
    __syncthreads();
    if (a.inputs_ready) {
        const unsigned char* src = reinterpret_cast<const unsigned char*>(bank) + (int64_t)c0 * ES;
        const int64_t rowb = (int64_t)hd * ES;
        const int lines = (int)((row_bytes + 127) >> 7);
        for (int i = tid; i < NR * lines; i += nt) {
            const int e = i / lines, l = i - e * lines;
            if (slot[e] >= 0) asm volatile("prefetch.global.L2 [%0];" ::"l"(src + slot[e] * rowb + (int64_t)l * 128));
        }
        grid_dependency_wait();
        if (early_trigger) grid_launch_dependents();
    }

    if (BULK) {
        // every thread: 16-byte cp.async copies of the entry row slices (zeros for skipped entries)
        const int cpr = (int)(row_bytes >> 4);
        unsigned char* dst = reinterpret_cast<unsigned char*>(rows);
        const unsigned char* src = reinterpret_cast<const unsigned char*>(bank) + (int64_t)c0 * ES;
        const size_t rs = (size_t)sw * ES;
        const int64_t rowb = (int64_t)hd * ES;
        const auto copy_chunk = [&](int e, int k) {
            const int64_t sl = slot[e];
            unsigned char* d = dst + e * rs + k * 16;
            if (sl >= 0)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(d)), "l"(src + sl * rowb + k * 16)
                             : "memory");
            else
                *reinterpret_cast<uint4*>(d) = make_uint4(0u, 0u, 0u, 0u);
        };
        if (nt % cpr == 0) {  // each thread keeps one 16-byte column of the rows
            const int k = tid % cpr, step = nt / cpr;
            for (int e = tid / cpr; e < NR; e += step) copy_chunk(e, k);
        } else {
            for (int c = tid; c < NR * cpr; c += nt) copy_chunk(c / cpr, c % cpr);
        }
        asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
        if (compact != nullptr) {  // this thread's own landed pieces of operand 0's named rows
            const auto put = [&](int e, int k) {
                if (kp[e] >= 0)
                    *reinterpret_cast<uint4*>(reinterpret_cast<unsigned char*>(compact) + kp[e] * rowb + c0 * ES +
                                              k * 16) = *reinterpret_cast<const uint4*>(dst + e * rs + k * 16);
            };
            if (nt % cpr == 0) {
                const int k = tid % cpr, step = nt / cpr;
                for (int e = tid / cpr; e < W0; e += step) put(e, k);
            } else {
                for (int c = tid; c < W0 * cpr; c += nt) put(c / cpr, c % cpr);
            }
        }
        fence_proxy_async_shared();  // the rows are read by bulk stores (async proxy) below
        __syncthreads();
        // stash: raw rows of operand 0 straight from shared memory
        if (stash_rows) {
            if (stash_bulk) {
                if (a.n_slices == 1) {
                    if (tid == 0) {
                        fence_proxy_async_shared();
                        bulk_s2g_hint(stash + t * W0 * hd, rows, (uint32_t)W0 * hd * ES, l2_evict_first());
                        bulk_commit();
                    }
                } else if (tid < 32) {
                    fence_proxy_async_shared();
                    for (int n = tid; n < W0; n += 32)
                        bulk_s2g(stash + (t * W0 + n) * hd + c0, rows + (size_t)n * sw, row_bytes);
                    bulk_commit();
                }
            } else if (active) {
                for (int n = 0; n < W0; ++n) stash[(t * W0 + n) * hd + c0 + j] = rows[(size_t)n * sw + j];
            }
        }
    } else if (active) {
        // plain loads of this thread's column; the bank is read-only for the kernel's lifetime
        int e = 0;
        for (; e + 8 <= NR; e += 8) {
            E x[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int64_t sl = slot[e + u];
                x[u] = sl >= 0 ? __ldg(bank + sl * hd + c0 + j) : E(0);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) rows[(size_t)(e + u) * sw + j] = x[u];
        }
        for (; e < NR; ++e) {
            const int64_t sl = slot[e];
            rows[(size_t)e * sw + j] = sl >= 0 ? __ldg(bank + sl * hd + c0 + j) : E(0);
        }
        if (compact != nullptr) {
            for (int n = 0; n < W0; ++n)
                if (kp[n] >= 0) compact[(int64_t)kp[n] * hd + c0 + j] = rows[(size_t)n * sw + j];
        } else if (stash_rows) {
            for (int n = 0; n < W0; ++n) stash[(t * W0 + n) * hd + c0 + j] = rows[(size_t)n * sw + j];
        }
    }

    // the weighted sum, one fmaf chain per column over ascending entries; bf16 rows and weights in
    // the full 128-column slice take two columns per thread (the first half of the threads):
    // compact snapshot 0.2764 -> 0.2725 ms, outputs only 0.2231 -> 0.2171 ms, the same bits
    if constexpr (kRawWeights<E, WT> && SW == kFullSlice) {
        const int p = 2 * tid;  // this thread's column pair (ncols is a multiple of 8)
        if (p < ncols) {
            const float2 r = weighted_sum_pair_bf16<SW>(reinterpret_cast<const uint16_t*>(rows) + p, wt, NR);
            float* o = a.out[op] + t * hd + c0 + p;
            if ((reinterpret_cast<uintptr_t>(o) & 7u) == 0) {
                *reinterpret_cast<float2*>(o) = r;
            } else {
                o[0] = r.x;
                o[1] = r.y;
            }
        }
    } else if (active) {
        a.out[op][t * hd + c0 + j] = weighted_sum<E, WT>(rows + j, sw, wt, NR);
    }
    // shared memory must outlive the bulk stores that read it
    if (BULK && stash_rows && stash_bulk && (a.n_slices == 1 ? tid == 0 : tid < 32)) bulk_wait_read_all();
}

template <typename E, typename I, typename WT>
void resolve_typed(bool bulk, GatherLaunch* L) {
    const auto kernel = !bulk ? gather_kernel<E, I, WT, false, 0>
                        : L->a.slice_cols == kFullSlice ? gather_kernel<E, I, WT, true, kFullSlice>
                                                        : gather_kernel<E, I, WT, true, 0>;
    L->fn = reinterpret_cast<const void*>(kernel);
}

template <typename E, typename I>
void resolve_w(int w_dtype, bool bulk, GatherLaunch* L) {
    if (w_dtype == SDM_BF16)
        resolve_typed<E, I, uint16_t>(bulk, L);
    else
        resolve_typed<E, I, float>(bulk, L);
}

int shrink_cols(int sw, bool bulk, int es) {
    const int q = bulk ? 16 / es : 32;
    const int half = (sw / 2 + q - 1) / q * q;
    return std::max(q, half);
}

}  // namespace

int plan_gather(const GatherArgs& a0, int bank_dtype, int idx_dtype, int w_dtype, GatherLaunch* L) {
    *L = GatherLaunch{};
    L->a = a0;
    GatherArgs& a = L->a;
    if (a.tokens == 0) return 0;
    const int es = bank_dtype == SDM_BF16 ? 2 : 4;
    // 16-byte row pieces: whole rows of 16-byte multiples, an aligned bank, and for a compact
    // snapshot (stored piece by piece) an aligned snapshot
    const bool bulk = ((int64_t)a.hd * es) % 16 == 0 && reinterpret_cast<uintptr_t>(a.bank) % 16 == 0 &&
                      (a.kpos == nullptr || reinterpret_cast<uintptr_t>(a.stash) % 16 == 0);
    const int n_rows = std::max(a.width[0], a.n_ops == 2 ? a.width[1] : 0);  // rows of one block

    int sw = std::min(a.hd, kMaxThreads);  // one column per thread
    if (bulk) sw = sw / (16 / es) * (16 / es);
    while ((size_t)n_rows * sw * es > kRowsBudget && sw > (bulk ? 16 / es : 32)) sw = shrink_cols(sw, bulk, es);
    a.slice_cols = sw;
    a.n_slices = (a.hd + sw - 1) / sw;
    const int64_t blocks = a.tokens * a.n_slices * a.n_ops;
    if (blocks > INT_MAX) return SDM_ECOUNT;
    L->stash_bulk =
        a.stash != nullptr && a.kpos == nullptr && reinterpret_cast<uintptr_t>(a.stash) % 16 == 0 && bulk;
    L->grid = (unsigned)blocks;
    L->block = (unsigned)((sw + 31) / 32 * 32);
    L->smem = GatherLayout(n_rows, sw, es).total;  // the wider operand's rows
    if (bank_dtype == SDM_BF16) {
        if (idx_dtype == SDM_I32)
            resolve_w<uint16_t, int32_t>(w_dtype, bulk, L);
        else
            resolve_w<uint16_t, int64_t>(w_dtype, bulk, L);
    } else {
        if (idx_dtype == SDM_I32)
            resolve_w<float, int32_t>(w_dtype, bulk, L);
        else
            resolve_w<float, int64_t>(w_dtype, bulk, L);
    }
    // the early trigger only when every block of this launch is resident at once; the shared-memory
    // limit is raised first, so that the occupancy query sees the launch's own limit
    const int rc = allow_smem(L->fn, L->smem);
    if (rc != 0) {
        *L = GatherLaunch{};
        return rc;
    }
    L->early_trigger = blocks <= (int64_t)blocks_per_sm(L->fn, (int)L->block, L->smem) * sm_count() ? 1 : 0;
    return 0;
}

int run_gather(const GatherLaunch& L, cudaStream_t stream) {
    if (L.fn == nullptr) return 0;
    GatherArgs a = L.a;
    int stash_bulk = L.stash_bulk, early = L.early_trigger;
    void* args[] = {&a, &stash_bulk, &early};
    return launch_pdl_raw(L.fn, dim3(L.grid), dim3(L.block), L.smem, stream, args);
}

int launch_gather(const GatherArgs& a, int bank_dtype, int idx_dtype, int w_dtype, cudaStream_t stream) {
    GatherLaunch L;
    const int rc = plan_gather(a, bank_dtype, idx_dtype, w_dtype, &L);
    if (rc != 0) return rc;
    return run_gather(L, stream);
}

int gather_status(unsigned int* word, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(word, g_gather_status, sizeof(unsigned int));
    if (e == cudaSuccess && clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_gather_status, &zero, sizeof(unsigned int));
    }
    return (int)e;
}

}  // namespace sdm
