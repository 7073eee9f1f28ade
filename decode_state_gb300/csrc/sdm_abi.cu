// C ABI of the SDM library: argument validation (host only, before any CUDA call) and dispatch to
// the kernel files. Every entry point follows include/sdm.h: 0 = launched, < 0 = argument error,
// > 0 = cudaError_t.
#include <atomic>
#include <climits>
#include <cstring>
#include <mutex>
#include <vector>

#include "sdm.h"
#include "sdm_internal.h"

namespace sdm {

int sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 148;
    }
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        n = 148;
    }
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

namespace {

// A device attribute of the current device, cached per device; `fallback` when it cannot be read.
int device_attribute(std::atomic<int>* cache, cudaDeviceAttr attr, int fallback) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return fallback;
    }
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, attr, dev) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        return fallback;
    }
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace

size_t smem_per_sm() {
    static std::atomic<int> cache[64];
    return (size_t)device_attribute(cache, cudaDevAttrMaxSharedMemoryPerMultiprocessor, 228 * 1024);
}

size_t smem_reserved_per_block() {
    static std::atomic<int> cache[64];
    return (size_t)device_attribute(cache, cudaDevAttrReservedSharedMemoryPerBlock, 1024);
}

int allow_smem(const void* kernel, size_t smem) {
    if (smem <= 48 * 1024) return 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return (int)e;
    }
    struct Raised {
        const void* fn;
        int dev;
        size_t bytes;
    };
    static std::mutex mu;
    static std::vector<Raised> raised;  // one entry per (kernel, device) raised so far
    std::lock_guard<std::mutex> lock(mu);
    Raised* r = nullptr;
    for (Raised& x : raised)
        if (x.fn == kernel && x.dev == dev) r = &x;
    if (r != nullptr && r->bytes >= smem) return 0;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return (int)e;
    }
    if (r != nullptr)
        r->bytes = smem;
    else
        raised.push_back(Raised{kernel, dev, smem});
    return 0;
}

int blocks_per_sm(const void* kernel, int threads, size_t smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    struct Entry {
        const void* fn;
        int dev, threads;
        size_t smem;
        int per_sm;
    };
    thread_local Entry cache[16] = {};
    thread_local unsigned next = 0;
    for (const Entry& x : cache)
        if (x.fn == kernel && x.dev == dev && x.threads == threads && x.smem == smem) return x.per_sm;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    cache[next++ % 16] = Entry{kernel, dev, threads, smem, n};
    return n;
}

}  // namespace sdm

namespace {

bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

bool overlaps(const void* a, size_t an, const void* b, size_t bn) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + bn && y < x + an;
}

int check_decode(void* bank, const void* k_idx, const float* k_val, const float* v, const float* beta,
                 const float* g, const void* q_idx, const float* q_val, void* out, int64_t n_streams, int hd, int W,
                 int R, int G, int T, int bank_dtype, int idx_dtype) {
    if (bank_dtype != SDM_BF16 && bank_dtype != SDM_F32) return SDM_EDTYPE;
    if (idx_dtype != SDM_I32 && idx_dtype != SDM_I64) return SDM_EIDX;
    if (hd < 1 || hd > 65536) return SDM_EHD;
    if (W < 1 || W > 256 || R < 1 || R > 256) return SDM_EWIDTH;
    if (G != 1 && G != W) return SDM_EGATES;
    if (n_streams < 0 || T < 0 || n_streams > (int64_t)INT_MAX) return SDM_ECOUNT;
    if (n_streams == 0 || T == 0) return SDM_OK;
    if (!bank || !k_idx || !k_val || !v || !beta || !g || !q_idx || !q_val || !out) return SDM_ENULL;
    const size_t es = bank_dtype == SDM_BF16 ? 2 : 4, is = idx_dtype == SDM_I64 ? 8 : 4;
    if (!aligned(bank, es) || !aligned(out, es) || !aligned(k_idx, is) || !aligned(q_idx, is) || !aligned(k_val, 4) ||
        !aligned(v, 4) || !aligned(beta, 4) || !aligned(g, 4) || !aligned(q_val, 4))
        return SDM_EALIGN;
    return SDM_OK;
}

int decode_common(void* bank, const void* k_idx, const float* k_val, const float* v, const float* beta,
                  const float* g, const void* q_idx, const float* q_val, void* out, int64_t n_streams, int hd, int W,
                  int R, int G, int T, int bank_dtype, int idx_dtype, int inputs_ready, bool stream_major,
                  sdm_stream_t stream) {
    const int rc = check_decode(bank, k_idx, k_val, v, beta, g, q_idx, q_val, out, n_streams, hd, W, R, G, T,
                                bank_dtype, idx_dtype);
    if (rc != SDM_OK || n_streams == 0 || T == 0) return rc;
    sdm::DecodeArgs a{};
    a.bank = bank;
    a.k_idx = k_idx;
    a.k_val = k_val;
    a.v = v;
    a.beta = beta;
    a.g = g;
    a.q_idx = q_idx;
    a.q_val = q_val;
    a.out = out;
    a.n_streams = n_streams;
    a.hd = hd;
    a.W = W;
    a.R = R;
    a.G = G;
    a.T = T;
    a.tstride = stream_major ? 1 : n_streams;
    a.sstride = stream_major ? T : 1;
    a.inputs_ready = inputs_ready;
    return sdm::launch_decode(a, bank_dtype, idx_dtype, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

int sdm_decode_seq(void* bank, const void* k_idx, const float* k_val, const float* v, const float* beta,
                   const float* g, const void* q_idx, const float* q_val, void* out, int64_t n_streams, int hd,
                   int W, int R, int G, int T, int bank_dtype, int idx_dtype, sdm_stream_t stream) {
    return decode_common(bank, k_idx, k_val, v, beta, g, q_idx, q_val, out, n_streams, hd, W, R, G, T, bank_dtype,
                         idx_dtype, 0, false, stream);
}

int sdm_decode_seq_ex(void* bank, const void* k_idx, const float* k_val, const float* v, const float* beta,
                      const float* g, const void* q_idx, const float* q_val, void* out, int64_t n_streams, int hd,
                      int W, int R, int G, int T, int bank_dtype, int idx_dtype, unsigned flags, sdm_stream_t stream) {
    if (flags & ~(SDM_INPUTS_READY | SDM_STREAM_MAJOR)) return SDM_EFLAGS;
    return decode_common(bank, k_idx, k_val, v, beta, g, q_idx, q_val, out, n_streams, hd, W, R, G, T, bank_dtype,
                         idx_dtype, (flags & SDM_INPUTS_READY) ? 1 : 0, (flags & SDM_STREAM_MAJOR) != 0, stream);
}

int sdm_decode_step(void* bank, const void* k_idx, const float* k_val, const float* v, const float* beta,
                    const float* g, const void* q_idx, const float* q_val, void* out, int64_t n_streams, int hd,
                    int W, int R, int G, int bank_dtype, int idx_dtype, sdm_stream_t stream) {
    return decode_common(bank, k_idx, k_val, v, beta, g, q_idx, q_val, out, n_streams, hd, W, R, G, 1, bank_dtype,
                         idx_dtype, 0, false, stream);
}

int sdm_decode_step_ex(void* bank, const void* k_idx, const float* k_val, const float* v, const float* beta,
                       const float* g, const void* q_idx, const float* q_val, void* out, int64_t n_streams, int hd,
                       int W, int R, int G, int bank_dtype, int idx_dtype, unsigned flags, sdm_stream_t stream) {
    if (flags & ~SDM_INPUTS_READY) return SDM_EFLAGS;
    return decode_common(bank, k_idx, k_val, v, beta, g, q_idx, q_val, out, n_streams, hd, W, R, G, 1, bank_dtype,
                         idx_dtype, (flags & SDM_INPUTS_READY) ? 1 : 0, false, stream);
}

}  // extern "C"

namespace {

// Shared validation of the gather entry points; fills *a when the arguments pass (SDM_OK). `stash`
// is the stash, or the compact snapshot when kpos is set (same byte size: tokens * width[0] rows).
int check_gather(const void* bank, int64_t n_slots, int hd, int bank_dtype, int n_ops, const void* const idx[2],
                 const void* const w[2], float* const out[2], const int width[2], int idx_dtype, int w_dtype,
                 void* stash, const int32_t* kpos, bool compact, int64_t tokens, int chunk, int valid,
                 const int32_t* chunk_valid, sdm::GatherArgs* a) {
    *a = sdm::GatherArgs{};
    if (bank_dtype != SDM_BF16 && bank_dtype != SDM_F32) return SDM_EDTYPE;
    if (w_dtype != SDM_BF16 && w_dtype != SDM_F32) return SDM_EDTYPE;
    if (idx_dtype != SDM_I32 && idx_dtype != SDM_I64) return SDM_EIDX;
    if (hd < 1 || hd > 65536) return SDM_EHD;
    if (n_ops != 1 && n_ops != 2) return SDM_ENOPS;
    if (!idx || !w || !out || !width) return SDM_ENULL;
    for (int o = 0; o < n_ops; ++o)
        if (width[o] < 1 || width[o] > 256) return SDM_EWIDTH;
    if (n_slots < 1 || n_slots > (int64_t)INT_MAX || tokens < 0 || tokens > (int64_t)INT_MAX) return SDM_ECOUNT;
    if (chunk < 1 || tokens % chunk != 0) return SDM_ECHUNK;
    if (chunk_valid == nullptr && (valid < 0 || valid > chunk)) return SDM_ECHUNK;
    if (tokens == 0) {
        a->chunk = chunk;
        return SDM_OK;
    }
    if (!bank) return SDM_ENULL;
    if (compact && (!stash || !kpos)) return SDM_ENULL;
    for (int o = 0; o < n_ops; ++o)
        if (!idx[o] || !w[o] || !out[o]) return SDM_ENULL;
    const size_t es = bank_dtype == SDM_BF16 ? 2 : 4, is = idx_dtype == SDM_I64 ? 8 : 4,
                 ws = w_dtype == SDM_BF16 ? 2 : 4;
    if (!aligned(bank, es) || (stash && !aligned(stash, es)) || (chunk_valid && !aligned(chunk_valid, 4)) ||
        (kpos && !aligned(kpos, 4)))
        return SDM_EALIGN;
    for (int o = 0; o < n_ops; ++o)
        if (!aligned(idx[o], is) || !aligned(w[o], ws) || !aligned(out[o], 4)) return SDM_EALIGN;
    const size_t bank_bytes = (size_t)n_slots * hd * es;
    for (int o = 0; o < n_ops; ++o)
        if (overlaps(out[o], (size_t)tokens * hd * 4, bank, bank_bytes)) return SDM_EOVERLAP;
    if (stash && overlaps(stash, (size_t)tokens * width[0] * hd * es, bank, bank_bytes)) return SDM_EOVERLAP;

    a->bank = bank;
    a->n_slots = n_slots;
    a->hd = hd;
    a->n_ops = n_ops;
    for (int o = 0; o < n_ops; ++o) {
        a->idx[o] = idx[o];
        a->w[o] = w[o];
        a->out[o] = out[o];
        a->width[o] = width[o];
    }
    a->stash = stash;
    a->kpos = compact ? kpos : nullptr;
    a->tokens = tokens;
    a->chunk = chunk;
    a->valid = valid;
    a->chunk_valid = chunk_valid;
    return SDM_OK;
}

int gather_common(const void* bank, int64_t n_slots, int hd, int bank_dtype, int n_ops, const void* const idx[2],
                  const void* const w[2], float* const out[2], const int width[2], int idx_dtype, int w_dtype,
                  void* stash, const int32_t* kpos, bool compact, int64_t tokens, int chunk, int valid,
                  const int32_t* chunk_valid, sdm_stream_t stream) {
    sdm::GatherArgs a;
    const int rc = check_gather(bank, n_slots, hd, bank_dtype, n_ops, idx, w, out, width, idx_dtype, w_dtype, stash,
                                kpos, compact, tokens, chunk, valid, chunk_valid, &a);
    if (rc != SDM_OK || tokens == 0) return rc;
    return sdm::launch_gather(a, bank_dtype, idx_dtype, w_dtype, reinterpret_cast<cudaStream_t>(stream));
}

// The contents of an sdm_gather_plan record. The tag mixes in an address inside this library, so a
// record made by another load of the library (whose kernel addresses differ) is refused.
struct PlanRecord {
    uint64_t tag;
    uint64_t bytes;
    int64_t row0_max;
    int64_t idx_row_bytes[2], w_row_bytes[2];  // bytes per index / weight row of each operand
    int32_t device, chunk;
    sdm::GatherLaunch launch;  // the launch at row0 = 0, valid = chunk
};
static_assert(sizeof(PlanRecord) <= SDM_GATHER_PLAN_BYTES, "gather plan record too large");

uint64_t plan_tag() {
    return 0x4e414c5047534453ull ^ (uint64_t)reinterpret_cast<uintptr_t>(&check_gather);
}

// The contents of an sdm_decode_plan record: the launch of token 0 and the byte step of every
// per-token array from one token to the next (time-major: n_streams rows per token).
struct DecodePlanRecord {
    uint64_t tag;
    uint64_t bytes;
    int64_t step[8];  // k_idx, k_val, v, beta, g, q_idx, q_val, out
    int32_t device, T;
    sdm::DecodeLaunch launch;  // token 0; nullptr kernel: nothing to launch
};
static_assert(sizeof(DecodePlanRecord) <= SDM_DECODE_PLAN_BYTES, "decode plan record too large");

uint64_t decode_plan_tag() {
    return 0x4e414c50434544ull ^ (uint64_t)reinterpret_cast<uintptr_t>(&check_decode);
}

}  // namespace

extern "C" {

int sdm_decode_plan_init(sdm_decode_plan* plan, void* bank, const void* k_idx, const float* k_val, const float* v,
                         const float* beta, const float* g, const void* q_idx, const float* q_val, void* out,
                         int64_t n_streams, int hd, int W, int R, int G, int T, int bank_dtype, int idx_dtype) {
    if (!plan) return SDM_ENULL;
    const int rc = check_decode(bank, k_idx, k_val, v, beta, g, q_idx, q_val, out, n_streams, hd, W, R, G, T,
                                bank_dtype, idx_dtype);
    if (rc != SDM_OK) return rc;
    DecodePlanRecord p{};
    const int64_t is = idx_dtype == SDM_I64 ? 8 : 4, es = bank_dtype == SDM_BF16 ? 2 : 4;
    const int64_t per[8] = {W * is, W * 4, (int64_t)hd * 4, 4, (int64_t)G * 4, R * is, R * 4, (int64_t)hd * es};
    for (int k = 0; k < 8; ++k) p.step[k] = per[k] * n_streams;
    p.T = T;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return (int)e;
    }
    p.device = dev;
    if (n_streams > 0 && T > 0) {
        sdm::DecodeArgs a{};
        a.bank = bank;
        a.k_idx = k_idx;
        a.k_val = k_val;
        a.v = v;
        a.beta = beta;
        a.g = g;
        a.q_idx = q_idx;
        a.q_val = q_val;
        a.out = out;
        a.n_streams = n_streams;
        a.hd = hd;
        a.W = W;
        a.R = R;
        a.G = G;
        a.T = 1;
        a.tstride = n_streams;
        a.sstride = 1;
        const int lrc = sdm::plan_decode(a, bank_dtype, idx_dtype, &p.launch);
        if (lrc != 0) return lrc;
    }
    p.tag = decode_plan_tag();
    p.bytes = sizeof(DecodePlanRecord);
    static_assert(sizeof(sdm_decode_plan) == SDM_DECODE_PLAN_BYTES, "decode plan record size");
    std::memset(plan, 0, sizeof(sdm_decode_plan));
    std::memcpy(plan, &p, sizeof(p));
    return SDM_OK;
}

int sdm_decode_plan_launch(const sdm_decode_plan* plan, int t, unsigned flags, sdm_stream_t stream) {
    return sdm_decode_plan_walk(plan, t, 1, flags, stream);
}

int sdm_decode_plan_walk(const sdm_decode_plan* plan, int t0, int n, unsigned flags, sdm_stream_t stream) {
    if (flags & ~SDM_INPUTS_READY) return SDM_EFLAGS;
    if (!plan) return SDM_ENULL;
    if (n < 0) return SDM_ECOUNT;
    DecodePlanRecord p;
    std::memcpy(&p, plan, sizeof(p));
    if (p.tag != decode_plan_tag() || p.bytes != sizeof(DecodePlanRecord)) return SDM_EPLAN;
    if (n > 0 && (t0 < 0 || (int64_t)t0 + n > p.T)) return SDM_EROW;
    if (p.launch.fn == nullptr || n == 0) return SDM_OK;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return SDM_EDEVICE;
    }
    if (dev != p.device) return SDM_EDEVICE;
    const sdm::DecodeArgs base = p.launch.a;
    sdm::DecodeArgs& a = p.launch.a;
    a.inputs_ready = (flags & SDM_INPUTS_READY) ? 1 : 0;
    const auto at = [](const void* q, int64_t off) { return static_cast<const unsigned char*>(q) + off; };
    for (int i = 0; i < n; ++i) {
        const int64_t t = (int64_t)t0 + i;
        a.k_idx = at(base.k_idx, t * p.step[0]);
        a.k_val = reinterpret_cast<const float*>(at(base.k_val, t * p.step[1]));
        a.v = reinterpret_cast<const float*>(at(base.v, t * p.step[2]));
        a.beta = reinterpret_cast<const float*>(at(base.beta, t * p.step[3]));
        a.g = reinterpret_cast<const float*>(at(base.g, t * p.step[4]));
        a.q_idx = at(base.q_idx, t * p.step[5]);
        a.q_val = reinterpret_cast<const float*>(at(base.q_val, t * p.step[6]));
        a.out = static_cast<unsigned char*>(base.out) + t * p.step[7];
        const int rc = sdm::run_decode(p.launch, reinterpret_cast<cudaStream_t>(stream));
        if (rc != 0) return rc;
    }
    return SDM_OK;
}

int sdm_gather(const void* bank, int64_t n_slots, int hd, int bank_dtype, int n_ops, const void* const idx[2],
               const void* const w[2], float* const out[2], const int width[2], int idx_dtype, int w_dtype,
               void* stash, int64_t tokens, int chunk, int valid, const int32_t* chunk_valid, sdm_stream_t stream) {
    return gather_common(bank, n_slots, hd, bank_dtype, n_ops, idx, w, out, width, idx_dtype, w_dtype, stash,
                         nullptr, false, tokens, chunk, valid, chunk_valid, stream);
}

int sdm_gather_kpos(const void* bank, int64_t n_slots, int hd, int bank_dtype, int n_ops, const void* const idx[2],
                    const void* const w[2], float* const out[2], const int width[2], int idx_dtype, int w_dtype,
                    void* compact, const int32_t* kpos, int64_t tokens, int chunk, int valid,
                    const int32_t* chunk_valid, sdm_stream_t stream) {
    return gather_common(bank, n_slots, hd, bank_dtype, n_ops, idx, w, out, width, idx_dtype, w_dtype, compact,
                         kpos, true, tokens, chunk, valid, chunk_valid, stream);
}

int sdm_gather_plan_init(sdm_gather_plan* plan, const void* bank, int64_t n_slots, int hd, int bank_dtype, int n_ops,
                         const void* const idx[2], const void* const w[2], float* const out[2], const int width[2],
                         int idx_dtype, int w_dtype, int64_t rows, int64_t row0_max, int64_t tokens, int chunk) {
    if (!plan) return SDM_ENULL;
    sdm::GatherArgs a;
    int rc = check_gather(bank, n_slots, hd, bank_dtype, n_ops, idx, w, out, width, idx_dtype, w_dtype, nullptr,
                          nullptr, false, tokens, chunk, chunk, nullptr, &a);
    if (rc != SDM_OK) return rc;
    if (row0_max < 0 || rows < tokens || row0_max > rows - tokens) return SDM_EROW;
    PlanRecord p{};
    const int64_t is = idx_dtype == SDM_I64 ? 8 : 4, ws = w_dtype == SDM_BF16 ? 2 : 4;
    for (int o = 0; o < n_ops; ++o) {
        p.idx_row_bytes[o] = is * width[o];
        p.w_row_bytes[o] = ws * width[o];
    }
    p.row0_max = row0_max;
    p.chunk = chunk;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return (int)e;
    }
    p.device = dev;
    if (tokens > 0) {
        rc = sdm::plan_gather(a, bank_dtype, idx_dtype, w_dtype, &p.launch);
        if (rc != 0) return rc;
    }
    p.tag = plan_tag();
    p.bytes = sizeof(PlanRecord);
    static_assert(sizeof(sdm_gather_plan) == SDM_GATHER_PLAN_BYTES, "plan record size");
    std::memset(plan, 0, sizeof(sdm_gather_plan));
    std::memcpy(plan, &p, sizeof(p));
    return SDM_OK;
}

int sdm_gather_plan_launch(const sdm_gather_plan* plan, int64_t row0, int valid, sdm_stream_t stream) {
    return sdm_gather_plan_launch_ex(plan, row0, valid, 0u, stream);
}

int sdm_gather_plan_launch_ex(const sdm_gather_plan* plan, int64_t row0, int valid, unsigned flags,
                              sdm_stream_t stream) {
    const int32_t v = valid;
    return sdm_gather_plan_walk(plan, &row0, &v, 1, flags, stream);
}

int sdm_gather_plan_walk(const sdm_gather_plan* plan, const int64_t* row0, const int32_t* valid, int n,
                         unsigned flags, sdm_stream_t stream) {
    if (flags & ~SDM_INPUTS_READY) return SDM_EFLAGS;
    if (!plan || (n > 0 && !row0)) return SDM_ENULL;
    if (n < 0) return SDM_ECOUNT;
    PlanRecord p;
    std::memcpy(&p, plan, sizeof(p));
    if (p.tag != plan_tag() || p.bytes != sizeof(PlanRecord)) return SDM_EPLAN;
    for (int i = 0; i < n; ++i)
        if (row0[i] < 0 || row0[i] > p.row0_max) return SDM_EROW;
    if (valid)
        for (int i = 0; i < n; ++i)
            if (valid[i] < 0 || valid[i] > p.chunk) return SDM_ECHUNK;
    if (p.launch.fn == nullptr || n == 0) return SDM_OK;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return SDM_EDEVICE;
    }
    if (dev != p.device) return SDM_EDEVICE;
    const sdm::GatherArgs base = p.launch.a;
    sdm::GatherArgs& a = p.launch.a;
    a.inputs_ready = (flags & SDM_INPUTS_READY) ? 1 : 0;
    for (int i = 0; i < n; ++i) {
        for (int o = 0; o < a.n_ops; ++o) {
            a.idx[o] = static_cast<const unsigned char*>(base.idx[o]) + row0[i] * p.idx_row_bytes[o];
            a.w[o] = static_cast<const unsigned char*>(base.w[o]) + row0[i] * p.w_row_bytes[o];
        }
        a.valid = valid ? valid[i] : p.chunk;
        const int rc = sdm::run_gather(p.launch, reinterpret_cast<cudaStream_t>(stream));
        if (rc != 0) return rc;
    }
    return SDM_OK;
}

const char* sdm_status_string(int status) {
    switch (status) {
        case SDM_OK: return "ok";
        case SDM_ENULL: return "a required pointer is NULL";
        case SDM_EDTYPE: return "bank or weight dtype must be SDM_BF16 or SDM_F32";
        case SDM_EIDX: return "index dtype must be SDM_I32 or SDM_I64";
        case SDM_EHD: return "head_dim must be in 1..65536";
        case SDM_EWIDTH: return "W, R and gather widths must be in 1..256";
        case SDM_EGATES: return "G must be 1 or W";
        case SDM_ECOUNT: return "a count is negative or too large for one launch, or n_slots is outside 1..2^31-1";
        case SDM_ECHUNK: return "need chunk >= 1, tokens a multiple of chunk and 0 <= valid <= chunk";
        case SDM_EALIGN: return "a pointer is not aligned to its element size";
        case SDM_EOVERLAP: return "a gather output or the stash overlaps the bank";
        case SDM_ENOPS: return "the gather takes one or two operands";
        case SDM_EPLAN: return "not a plan made by sdm_gather_plan_init / sdm_decode_plan_init in this process";
        case SDM_EROW: return "row0 outside 0..row0_max, row0_max + tokens beyond the index rows, or a plan step outside 0..T-1";
        case SDM_EDEVICE: return "the current device is not the plan's device";
        case SDM_EFLAGS: return "unknown bits in the flags of an _ex entry point";
        default: break;
    }
    if (status > 0) return cudaGetErrorString(static_cast<cudaError_t>(status));
    return "unknown status";
}

int sdm_device_status(unsigned int* status, int clear) {
    if (!status) return SDM_ENULL;
    // every kernel of the device, on any stream, has finished before the words are read (and
    // cleared): the symbol copies below are ordered only on the legacy default stream
    const cudaError_t s = cudaDeviceSynchronize();
    if (s != cudaSuccess) {
        (void)cudaGetLastError();
        *status = 0;
        return (int)s;
    }
    unsigned int a = 0, b = 0;
    int e = sdm::decode_status(&a, clear != 0);
    if (e == 0) e = sdm::gather_status(&b, clear != 0);
    *status = a | b;
    if (e != 0) (void)cudaGetLastError();
    return e;
}

int sdm_version(void) { return 200; }

}  // extern "C"
