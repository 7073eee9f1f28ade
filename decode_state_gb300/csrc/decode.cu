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
// the reference kernel makes for its CTA barrier).
//
// Vector path (rows a multiple of 16 bytes), per token:
//   1. every thread issues 16-byte cp.async copies of the W write row slices into shared memory
//      (all in flight at once), L2 prefetches of this token's R read rows (only a hint: the
//      copies in step 3 still read the rows as the write left them, from L2), then cp.async
//      copies of the NEXT token's slots and weights, and thread 0 computes the next token's
//      shared gate;
//   2. each thread owns two adjacent columns, held as a packed float32 pair, and runs the
//      retrieve as one chain of paired fmas over ascending w, then delta, then the decay-and-write
//      (paired multiply and fma, one paired round to the bank dtype). With many blocks per SM the
//      owners publish their delta pairs and the write goes by 16-byte pieces instead (thread =
//      row group and piece, one 16-byte load and store per row it takes), which needs a quarter
//      of the per-row loads, stores and address work; otherwise each thread writes its own pair
//      of every row (the one-column kernel for narrow slices always writes by pieces);
//   3. a barrier, then the R read rows by 16-byte cp.async, and each thread reduces its columns
//      over ascending r (for bf16 banks with the mixed-precision fma, whose bf16 operands need no
//      widening); meanwhile the next token's write rows are prefetched into L2, so that its
//      copies in step 1 are served from L2 while their DRAM reads overlap this step;
//   4. the prefetched metadata of the next token is turned into row byte offsets and broadcast
//      weight pairs in shared memory (16-byte aligned arrays, read two rows' worth per load).
// The rows travel as 16-byte cp.async copies (the load/store path, generic proxy) rather than one
// bulk copy per row: with 256-byte rows the bulk-copy engine sustained about 3 TB/s of row reads
// per GPU, the 16-byte copies spread over all threads sustain the rest of HBM. Being generic-proxy
// copies, they see the block's earlier stores after a plain barrier, and no wait in this file
// spins.
// Rows that are not a multiple of 16 bytes (or unaligned pointers) take a plain-load path with
// one column per thread; a thread then only ever touches its own column, so program order alone
// orders its writes and reads.
//
// Arithmetic per element (float32; every paired op is two independent round-to-nearest ops):
//   a_w = kv_w * d_w;  retrieved = fma(a_w, row_w, .) over w;  delta = beta * (round(v) - retrieved)
//   new_w = fma(kv_w, delta, row_w * d_w);  readings = fma(qv_r, row_r, .) over r
// with d_w the float32 nearest to e^g (gate(): a float32-pair table evaluation kept when a rounding
// test proves it is that float32, the double-precision exponential rounded once otherwise).
#include <algorithm>
#include <climits>

#include "sdm.h"
#include "sdm_device.cuh"
#include "sdm_internal.h"

namespace sdm {
namespace {

__device__ unsigned int g_decode_status;

constexpr int kMaxThreads = 256;
constexpr size_t kRowsBudget = 32 * 1024;  // staged rows of one block; with the metadata this stays under 48 KB

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------- packed float32 pairs

__device__ __forceinline__ uint64_t f2(float lo, float hi) {
    return ((uint64_t)__float_as_uint(hi) << 32) | (uint64_t)__float_as_uint(lo);
}
__device__ __forceinline__ float f2lo(uint64_t x) { return __uint_as_float((uint32_t)x); }
__device__ __forceinline__ float f2hi(uint64_t x) { return __uint_as_float((uint32_t)(x >> 32)); }
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// ---------------------------------------------------------------- gates
//
// d = the float32 nearest to e^g, without the double-precision exponential in the common case.
// Tang's table method (P. T. P. Tang, "Table-driven implementation of the exponential function in
// IEEE floating-point arithmetic", ACM TOMS 15(2), 1989) in float32 pairs: g = (64m + j) ln2/64 + r
// with |r| <= 0.00543, and e^g = 2^m 2^(j/64) e^r, where e^r - 1 = r + r^2/2 + r^3 (1/6 + r/24 +
// r^2/120) truncates below 2^-54. The reduction is exact up to 2^-51 (ln2/64 = A + B + C with A of
// 9 bits, so nA is exact and g - nA exact; nB an exact product pair), the sum keeps r and r^2/2 as
// pairs, and the whole evaluation stays within 2^-42 of e^g. The pair is rounded once; the result
// is taken when the pair lies more than 2^-38 (in units of the scaled value, in [0.99, 2)) inside
// the rounding interval (Ziv's test, A. Ziv, ACM TOMS 17(3), 1991), and is then the float32 nearest
// to e^g -- the value that rounding the double-precision exponential gives, which is within 2^-51 of
// e^g. Otherwise (about one gate in 10^4) and outside [-87, 88] (subnormal, huge or NaN results)
// the double-precision exponential decides, so every gate has the bits of gate(g).

// 2^(j/64) = hi + lo (each the float32 nearest; the pair within 2^-49 of the power)
__device__ const float2 kExp2Tab[64] = {
    {0x1.0p0f, 0.0f}, {0x1.02c9a4p0f, -0x1.887fap-28f},
    {0x1.059b0ep0f, -0x1.9d4f52p-25f}, {0x1.087452p0f, -0x1.e2990ep-26f},
    {0x1.0b5586p0f, 0x1.9f3122p-25f}, {0x1.0e3ec4p0f, -0x1.a585ccp-25f},
    {0x1.11301ep0f, -0x1.fdb496p-25f}, {0x1.1429aap0f, 0x1.d525bcp-25f},
    {0x1.172b84p0f, -0x1.c15742p-27f}, {0x1.1a35bep0f, 0x1.6df96ep-25f},
    {0x1.1d4874p0f, -0x1.d2e8cap-25f}, {0x1.2063b8p0f, 0x1.0c519ap-25f},
    {0x1.2387a6p0f, 0x1.ceac48p-25f}, {0x1.26b456p0f, 0x1.789f38p-26f},
    {0x1.29e9ep0f, -0x1.5c0424p-25f}, {0x1.2d285ap0f, 0x1.b900c2p-26f},
    {0x1.306fep0f, 0x1.4636e2p-25f}, {0x1.33c08cp0f, -0x1.b37d2p-25f},
    {0x1.371a74p0f, -0x1.18aac6p-25f}, {0x1.3a7db4p0f, -0x1.634c02p-25f},
    {0x1.3dea64p0f, 0x1.824684p-25f}, {0x1.4160a2p0f, 0x1.f72e2ap-28f},
    {0x1.44e086p0f, 0x1.8624b4p-30f}, {0x1.486a2cp0f, -0x1.47d866p-25f},
    {0x1.4bfdaep0f, -0x1.593abcp-25f}, {0x1.4f9b28p0f, -0x1.2c5a6cp-25f},
    {0x1.5342b6p0f, -0x1.2c561p-25f}, {0x1.56f474p0f, -0x1.295b04p-25f},
    {0x1.5ab07ep0f, -0x1.5bd5ecp-27f}, {0x1.5e76f2p0f, -0x1.4a5bd6p-25f},
    {0x1.6247ecp0f, -0x1.f8b55p-25f}, {0x1.662388p0f, 0x1.2a9112p-27f},
    {0x1.6a09e6p0f, 0x1.9fcef4p-26f}, {0x1.6dfb24p0f, -0x1.cd72e8p-27f},
    {0x1.71f75ep0f, 0x1.1d8beep-25f}, {0x1.75feb6p0f, -0x1.37b306p-25f},
    {0x1.7a1148p0f, -0x1.829fdp-25f}, {0x1.7e2f34p0f, -0x1.261634p-25f},
    {0x1.82589ap0f, -0x1.accc7cp-26f}, {0x1.868d9ap0f, -0x1.2edb44p-26f},
    {0x1.8ace54p0f, 0x1.15506ep-27f}, {0x1.8f1aeap0f, -0x1.baa232p-26f},
    {0x1.93737cp0f, -0x1.e64744p-25f}, {0x1.97d82ap0f, -0x1.0d8d84p-31f},
    {0x1.9c4918p0f, 0x1.51f848p-27f}, {0x1.a0c668p0f, -0x1.2886a6p-26f},
    {0x1.a5503cp0f, -0x1.b83b54p-25f}, {0x1.a9e6b6p0f, -0x1.50c048p-25f},
    {0x1.ae89fap0f, -0x1.a94b14p-26f}, {0x1.b33a2cp0f, -0x1.ec3a82p-26f},
    {0x1.b7f77p0f, -0x1.a09438p-25f}, {0x1.bcc1eap0f, -0x1.f687c6p-25f},
    {0x1.c199bep0f, -0x1.3d56b2p-27f}, {0x1.c67f12p0f, 0x1.cafa2ap-25f},
    {0x1.cb720ep0f, -0x1.8837ccp-27f}, {0x1.d072d4p0f, 0x1.40f13p-25f},
    {0x1.d5818ep0f, -0x1.822dbcp-27f}, {0x1.da9e6p0f, 0x1.ed9942p-27f},
    {0x1.dfc974p0f, -0x1.908c94p-25f}, {0x1.e502eep0f, 0x1.e2cffep-26f},
    {0x1.ea4afap0f, 0x1.52486cp-27f}, {0x1.efa1bep0f, 0x1.cc2b44p-25f},
    {0x1.f50766p0f, -0x1.246ebp-26f}, {0x1.fa7c18p0f, 0x1.9e90d8p-28f},
};

// the error of s = a + b (rounded): a + b = s + two_sum_err(a, b, s) exactly
__device__ __forceinline__ float two_sum_err(float a, float b, float s) {
    const float bb = __fsub_rn(s, a);
    return __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

__device__ __forceinline__ float gate(float g) {
    if (fabsf(g) < 0x1p-30f) return 1.0f;  // e^g within 2^-30 of 1, far from both rounding midpoints
    if (!(g >= -87.0f && g <= 88.0f)) return (float)exp((double)g);
    constexpr float kInv = 0x1.715476p6f;  // 64 / ln2
    constexpr float kA = 0x1.63p-7f, kB = -0x1.bd0106p-19f, kC = 0x1.cf79acp-46f;  // ln2/64 = A + B + C
    const float nf = rintf(__fmul_rn(g, kInv));  // |n| <= 8126
    const int n = (int)nf, j = n & 63, m = n >> 6;  // n = 64m + j, 0 <= j < 64
    const float t1 = fmaf(-nf, kA, g);               // g - nA, exact
    const float p_hi = __fmul_rn(nf, kB);
    const float p_lo = fmaf(nf, kB, -p_hi);          // nB = p_hi + p_lo exactly
    const float r_hi = __fsub_rn(t1, p_hi);
    const float r_lo = __fsub_rn(__fsub_rn(two_sum_err(t1, -p_hi, r_hi), p_lo), __fmul_rn(nf, kC));
    const float s_hi = __fmul_rn(r_hi, r_hi);
    const float s_lo = fmaf(r_hi, r_hi, -s_hi);      // r_hi^2 = s_hi + s_lo exactly
    const float h = __fmul_rn(0.5f, s_hi);
    const float u_hi = __fadd_rn(r_hi, h);
    const float cubic = __fmul_rn(__fmul_rn(r_hi, s_hi),
                                  fmaf(r_hi, fmaf(r_hi, 1.0f / 120.0f, 1.0f / 24.0f), 1.0f / 6.0f));
    const float low = two_sum_err(r_hi, h, u_hi) + r_lo + (0.5f * s_lo + r_hi * r_lo) + cubic;
    const float e_hi = __fadd_rn(1.0f, u_hi);        // e^r = e_hi + e_lo
    const float e_lo = __fadd_rn(__fadd_rn(__fsub_rn(1.0f, e_hi), u_hi), low);
    const float2 t = __ldg(&kExp2Tab[j]);
    const float y_hi = __fmul_rn(t.x, e_hi);         // 2^(j/64) e^r = y_hi + y_lo
    const float y_lo = fmaf(t.y, e_hi, fmaf(t.x, e_lo, fmaf(t.x, e_hi, -y_hi)));
    const float f = __fadd_rn(y_hi, y_lo);
    const float dev = __fadd_rn(__fsub_rn(y_hi, f), y_lo);  // (y_hi + y_lo) - f, to 2^-48
    const uint32_t fb = __float_as_uint(f);
    const float ulp = __uint_as_float((fb & 0x7f800000u) - (23u << 23));
    const float half = (dev < 0.0f && (fb & 0x007fffffu) == 0) ? 0.25f * ulp : 0.5f * ulp;
    if (fabsf(dev) < half - 0x1p-38f) return __uint_as_float(fb + ((uint32_t)m << 23));  // f 2^m, normal
    return (float)exp((double)g);
}

// lo += q * x.lo, hi += q * x.hi for a bf16 pair x, with q the bf16 held in the high half of the
// float32 bit pattern qbits (exact when the float32 is bf16-representable); one rounding each
__device__ __forceinline__ void fma_bf16_pair(float& lo, float& hi, uint32_t qbits, uint32_t x) {
    asm("{\n\t.reg .b16 xl, xh, ql, qh;\n\t"
        "mov.b32 {xl, xh}, %2;\n\t"
        "mov.b32 {ql, qh}, %3;\n\t"
        "fma.rn.f32.bf16 %0, qh, xl, %0;\n\t"
        "fma.rn.f32.bf16 %1, qh, xh, %1;\n\t}"
        : "+f"(lo), "+f"(hi)
        : "r"(x), "r"(qbits));
}

// two adjacent bank elements as one word, widened to / narrowed from a float32 pair
template <typename E>
struct Pair;
template <>
struct Pair<uint16_t> {
    using T = uint32_t;
    __device__ static __forceinline__ uint64_t widen(uint32_t u) {
        return f2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
    }
    __device__ static __forceinline__ uint32_t narrow(uint64_t x) {  // round to nearest even, both lanes
        __nv_bfloat162 h = __floats2bfloat162_rn(f2lo(x), f2hi(x));
        return *reinterpret_cast<uint32_t*>(&h);
    }
};
template <>
struct Pair<float> {
    using T = uint64_t;
    __device__ static __forceinline__ uint64_t widen(uint64_t u) { return u; }
    __device__ static __forceinline__ uint64_t narrow(uint64_t x) { return x; }
};

// ---------------------------------------------------------------- vector-path layout

struct VecLayout {
    size_t rows, raw_k, raw_kv, raw_g, raw_q, raw_qv, raw_beta, koff, qoff, aw2, kv2, dw2, qv2, beta, dnext, dlt, total;
    __host__ __device__ VecLayout(int W, int R, int G, int sw, int es, int is) {
        const int maxwr = W > R ? W : R;
        rows = 0;
        raw_k = align_up((size_t)maxwr * sw * es, 16);
        raw_kv = align_up(raw_k + (size_t)W * is, 16);
        raw_g = align_up(raw_kv + (size_t)W * 4, 16);
        raw_q = align_up(raw_g + (size_t)G * 4, 16);
        raw_qv = align_up(raw_q + (size_t)R * is, 16);
        raw_beta = align_up(raw_qv + (size_t)R * 4, 16);
        koff = align_up(raw_beta + 4, 16);
        qoff = align_up(koff + (size_t)W * 8, 16);
        aw2 = align_up(qoff + (size_t)R * 8, 16);
        kv2 = align_up(aw2 + (size_t)W * 8, 16);
        dw2 = align_up(kv2 + (size_t)W * 8, 16);
        qv2 = align_up(dw2 + (size_t)(G == 1 ? 1 : W) * 8, 16);  // one shared gate when G == 1
        beta = align_up(qv2 + (size_t)R * 8, 16);
        dnext = beta + 4;
        dlt = align_up(dnext + 4, 16);  // the delta pair of every column pair of the slice
        total = dlt + (size_t)(sw / 2) * 8;
    }
};

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Every thread: cp.async copies of token ts's slots, weights, gates and beta into the raw area.
template <typename I, typename Layout>
__device__ __forceinline__ void prefetch_meta(const DecodeArgs& a, int64_t ts, const Layout& L, unsigned char* smem) {
    const int tid = threadIdx.x, nt = blockDim.x, W = a.W, R = a.R, G = a.G;
    I* rk = reinterpret_cast<I*>(smem + L.raw_k);
    I* rq = reinterpret_cast<I*>(smem + L.raw_q);
    float* rkv = reinterpret_cast<float*>(smem + L.raw_kv);
    float* rg = reinterpret_cast<float*>(smem + L.raw_g);
    float* rqv = reinterpret_cast<float*>(smem + L.raw_qv);
    const I* k_idx = static_cast<const I*>(a.k_idx) + ts * W;
    const I* q_idx = static_cast<const I*>(a.q_idx) + ts * R;
    for (int i = tid; i < W; i += nt) {
        if constexpr (sizeof(I) == 8)
            cp_async8(rk + i, k_idx + i);
        else
            cp_async4(rk + i, k_idx + i);
        cp_async4(rkv + i, a.k_val + ts * W + i);
    }
    for (int i = tid; i < G; i += nt) cp_async4(rg + i, a.g + ts * G + i);
    for (int i = tid; i < R; i += nt) {
        if constexpr (sizeof(I) == 8)
            cp_async8(rq + i, q_idx + i);
        else
            cp_async4(rq + i, q_idx + i);
        cp_async4(rqv + i, a.q_val + ts * R + i);
    }
    if (tid == 0) cp_async4(smem + L.raw_beta, a.beta + ts);
    cp_async_commit();
}

// Every thread: turn the raw copies into row byte offsets and broadcast weight pairs.
template <typename E, typename I>
__device__ __forceinline__ void derive_meta(const DecodeArgs& a, int c0, const VecLayout& L, unsigned char* smem) {
    const int tid = threadIdx.x, nt = blockDim.x, W = a.W, R = a.R, G = a.G;
    const int64_t rowb = (int64_t)a.hd * sizeof(E), colb = (int64_t)c0 * sizeof(E);
    const I* rk = reinterpret_cast<const I*>(smem + L.raw_k);
    const I* rq = reinterpret_cast<const I*>(smem + L.raw_q);
    const float* rkv = reinterpret_cast<const float*>(smem + L.raw_kv);
    const float* rg = reinterpret_cast<const float*>(smem + L.raw_g);
    const float* rqv = reinterpret_cast<const float*>(smem + L.raw_qv);
    int64_t* koff = reinterpret_cast<int64_t*>(smem + L.koff);
    int64_t* qoff = reinterpret_cast<int64_t*>(smem + L.qoff);
    uint64_t* aw2 = reinterpret_cast<uint64_t*>(smem + L.aw2);
    uint64_t* kv2 = reinterpret_cast<uint64_t*>(smem + L.kv2);
    uint64_t* dw2 = reinterpret_cast<uint64_t*>(smem + L.dw2);
    uint64_t* qv2 = reinterpret_cast<uint64_t*>(smem + L.qv2);
    const float d1 = *reinterpret_cast<const float*>(smem + L.dnext);
    for (int i = tid; i < W; i += nt) {
        koff[i] = (int64_t)rk[i] * rowb + colb;
        const float k = round_to<E>(rkv[i]);
        const float d = G == 1 ? d1 : gate(rg[i]);
        const float aa = __fmul_rn(k, d);
        kv2[i] = f2(k, k);
        aw2[i] = f2(aa, aa);
        if (G != 1 || i == 0) dw2[i] = f2(d, d);
    }
    for (int i = tid; i < R; i += nt) {
        qoff[i] = (int64_t)rq[i] * rowb + colb;
        const float q = round_to<E>(rqv[i]);
        qv2[i] = f2(q, q);
    }
    if (tid == 0) *reinterpret_cast<float*>(smem + L.beta) = *reinterpret_cast<const float*>(smem + L.raw_beta);
}

// Every thread: 16-byte cp.async copies (LSU path, generic proxy) of n row slices at byte offsets
// off[] into rows[i * sw]; one commit group.
template <typename E>
__device__ __forceinline__ void ldgsts_rows(E* rows, const unsigned char* bank, const int64_t* off, int n, int sw,
                                            uint32_t row_bytes) {
    const int tid = threadIdx.x, nt = blockDim.x;
    const int cpr = (int)(row_bytes >> 4);  // 16-byte chunks per row slice
    unsigned char* dst = reinterpret_cast<unsigned char*>(rows);
    const size_t rs = (size_t)sw * sizeof(E);
    if (nt % cpr == 0) {
        const int k = tid % cpr, step = nt / cpr;
        for (int r = tid / cpr; r < n; r += step)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst + r * rs + k * 16)),
                         "l"(bank + off[r] + k * 16)
                         : "memory");
    } else {
        for (int c = tid; c < n * cpr; c += nt) {
            const int r = c / cpr, k = c - r * cpr;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst + r * rs + k * 16)),
                         "l"(bank + off[r] + k * 16)
                         : "memory");
        }
    }
    cp_async_commit();
}

// an L2 prefetch (a hint: nothing reaches the SM) of the 128-byte line at p
__device__ __forceinline__ void pf_l2(const void* p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

// L2 prefetches (hints: nothing reaches the SM) of the 128-byte lines of n row slices bank + off[r]
__device__ __forceinline__ void prefetch_rows_l2(const unsigned char* bank, const int64_t* off, int n,
                                                 uint32_t row_bytes) {
    const int lines = (int)((row_bytes + 127) >> 7);
    for (int i = threadIdx.x; i < n * lines; i += blockDim.x) {
        const int r = i / lines, l = i - r * lines;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(bank + off[r] + (int64_t)l * 128));
    }
}

// PIECE = false compiles the per-pair write-back only; the launcher takes the PIECE instances on
// every grid (the write-back by pieces measured faster at 2, 3, 4 and 7 blocks per SM), which
// still fall back to the per-pair path where the pieces do not tile the block's threads.
// SW (every kernel below): the slice width in columns when it is fixed at compile time, so that
// the staged rows' addresses in shared memory are immediate offsets; 0 takes it from the arguments.
template <typename E, typename I, bool PIECE, int SW = 0>
__global__ void __launch_bounds__(kMaxThreads, 2) decode_vec_kernel(const DecodeArgs a, int early_trigger) {
    using P = Pair<E>;
    using PT = typename P::T;
    constexpr int ES = sizeof(E);
    extern __shared__ __align__(128) unsigned char smem[];

    const int W = a.W, R = a.R, G = a.G, hd = a.hd, sw = SW ? SW : a.slice_cols;
    const VecLayout L(W, R, G, sw, ES, (int)sizeof(I));
    E* rows = reinterpret_cast<E*>(smem + L.rows);
    const int64_t* koff = reinterpret_cast<const int64_t*>(smem + L.koff);
    const int64_t* qoff = reinterpret_cast<const int64_t*>(smem + L.qoff);
    const uint64_t* aw2 = reinterpret_cast<const uint64_t*>(smem + L.aw2);
    const uint64_t* kv2 = reinterpret_cast<const uint64_t*>(smem + L.kv2);
    const uint64_t* dw2 = reinterpret_cast<const uint64_t*>(smem + L.dw2);
    const uint64_t* qv2 = reinterpret_cast<const uint64_t*>(smem + L.qv2);

    const int tid = threadIdx.x;
    const int64_t s = blockIdx.x / a.n_slices;
    const int c0 = (int)(blockIdx.x % a.n_slices) * sw;
    const int ncols = min(sw, hd - c0);
    const int j = 2 * tid;  // this thread's first column within the slice
    const bool active = j < ncols;
    const uint32_t row_bytes = (uint32_t)ncols * ES;
    const int pstride = sw / 2;  // pairs per staged row
    unsigned char* bank = static_cast<unsigned char*>(a.bank);
    E* out = static_cast<E*>(a.out);
    const PT* rp = reinterpret_cast<const PT*>(rows) + tid;
    const int64_t jb = (int64_t)j * ES;
    const int nt = blockDim.x;
    const int cpr = (int)(row_bytes >> 4);  // 16-byte pieces per row slice
    const bool by_piece = PIECE && a.piece_write && nt % cpr == 0 && nt / cpr <= W;

    // With inputs_ready the inputs predate the preceding kernel: token 0's metadata is read and its
    // rows are warmed in L2 before waiting for that kernel; the bank is read and written (and `out`
    // written) only after the wait. L2 is the point of coherence, so a line warmed early still
    // holds every later write to it. The next launch is released only after the wait, so at most
    // one launch runs its early part ahead of the kernel that is working.
    if (!a.inputs_ready) {
        grid_dependency_wait();
        if (early_trigger) grid_launch_dependents();
    }
    prefetch_meta<I>(a, s * a.sstride, L, smem);  // token 0
    cp_async_wait_all();
    __syncthreads();
    if (G == 1 && tid == 0)
        *reinterpret_cast<float*>(smem + L.dnext) = gate(*reinterpret_cast<const float*>(smem + L.raw_g));
    __syncthreads();
    derive_meta<E, I>(a, c0, L, smem);
    __syncthreads();
    if (a.inputs_ready) {
        prefetch_rows_l2(bank, koff, W, row_bytes);
        prefetch_rows_l2(bank, qoff, R, row_bytes);
        grid_dependency_wait();
        if (early_trigger) grid_launch_dependents();
    }

    for (int t = 0; t < a.T; ++t) {
        const int64_t ts = (int64_t)t * a.tstride + s * a.sstride;  // (token, stream) row of the inputs

        // 1. the write rows; the next token's metadata meanwhile
        ldgsts_rows<E>(rows, bank, koff, W, sw, row_bytes);
        {  // this token's read rows into L2 meanwhile: step 3 then copies them from L2
            const int lines = (int)((row_bytes + 127) >> 7);
            for (int i = tid; i < R * lines; i += blockDim.x) {
                const int r = i / lines, l = i - r * lines;
                pf_l2(bank + qoff[r] + (int64_t)l * 128);
            }
        }
        uint64_t vr = 0;
        if (active) {
            const float2 vv = __ldg(reinterpret_cast<const float2*>(a.v + ts * hd + c0 + j));
            vr = P::widen(P::narrow(f2(vv.x, vv.y)));  // rounded to the bank dtype
        }
        const float beta = *reinterpret_cast<const float*>(smem + L.beta);
        const uint64_t dsh = dw2[0];
        const bool more = t + 1 < a.T;
        if (more) {
            prefetch_meta<I>(a, ts + a.tstride, L, smem);
            if (G == 1 && tid == 0)  // the next token's shared gate, while this token's rows are in flight
                *reinterpret_cast<float*>(smem + L.dnext) = gate(__ldg(a.g + ts + a.tstride));
        }
        if (more)
            asm volatile("cp.async.wait_group 1;" ::: "memory");  // the rows, not yet the metadata
        else
            cp_async_wait_all();
        __syncthreads();

        // 2. retrieve, delta, decay-and-write
        if (active) {
            uint64_t acc = 0;
            int w = 0;
            for (; w + 4 <= W; w += 4) {
                const PT x0 = rp[(w + 0) * pstride], x1 = rp[(w + 1) * pstride];
                const PT x2 = rp[(w + 2) * pstride], x3 = rp[(w + 3) * pstride];
                const ulonglong2 a01 = *reinterpret_cast<const ulonglong2*>(aw2 + w);
                const ulonglong2 a23 = *reinterpret_cast<const ulonglong2*>(aw2 + w + 2);
                acc = ffma2(a01.x, P::widen(x0), acc);
                acc = ffma2(a01.y, P::widen(x1), acc);
                acc = ffma2(a23.x, P::widen(x2), acc);
                acc = ffma2(a23.y, P::widen(x3), acc);
            }
            for (; w < W; ++w) acc = ffma2(aw2[w], P::widen(rp[w * pstride]), acc);
            const float dl = __fmul_rn(beta, __fsub_rn(f2lo(vr), f2lo(acc)));
            const float dh = __fmul_rn(beta, __fsub_rn(f2hi(vr), f2hi(acc)));
            const uint64_t delta = f2(dl, dh);
            if (by_piece) {
                reinterpret_cast<uint64_t*>(smem + L.dlt)[tid] = delta;
            } else {  // each thread writes its own pair of every row
                unsigned char* bj = bank + jb;
                w = 0;
#pragma unroll 2
                for (; w + 2 <= W; w += 2) {
                    const uint64_t x0 = P::widen(rp[w * pstride]), x1 = P::widen(rp[(w + 1) * pstride]);
                    const ulonglong2 k2 = *reinterpret_cast<const ulonglong2*>(kv2 + w);
                    const longlong2 o2 = *reinterpret_cast<const longlong2*>(koff + w);
                    uint64_t d0 = dsh, d1 = dsh;
                    if (G != 1) {
                        const ulonglong2 dd = *reinterpret_cast<const ulonglong2*>(dw2 + w);
                        d0 = dd.x;
                        d1 = dd.y;
                    }
                    const uint64_t y0 = ffma2(k2.x, delta, fmul2(x0, d0));
                    const uint64_t y1 = ffma2(k2.y, delta, fmul2(x1, d1));
                    *reinterpret_cast<PT*>(bj + o2.x) = P::narrow(y0);
                    *reinterpret_cast<PT*>(bj + o2.y) = P::narrow(y1);
                }
                for (; w < W; ++w) {
                    const uint64_t x = P::widen(rp[w * pstride]);
                    const uint64_t y = ffma2(kv2[w], delta, fmul2(x, G == 1 ? dsh : dw2[w]));
                    *reinterpret_cast<PT*>(bj + koff[w]) = P::narrow(y);
                }
            }
        }
        if (by_piece) {
            // the decay-and-write by 16-byte pieces: thread = (row group, piece); every thread
            // takes one piece of every ngroups-th row, with the delta pairs its owners published
            __syncthreads();
            constexpr int PP = 16 / (2 * ES);  // column pairs per piece
            const int k = tid % cpr, ngroups = nt / cpr;
            uint64_t dp[PP];
#pragma unroll
            for (int p = 0; p < PP; ++p) dp[p] = reinterpret_cast<const uint64_t*>(smem + L.dlt)[k * PP + p];
            const unsigned char* src = reinterpret_cast<const unsigned char*>(rows) + k * 16;
            unsigned char* dst = bank + k * 16;
            const size_t rstride = (size_t)sw * ES;
#pragma unroll 2
            for (int w = tid / cpr; w < W; w += ngroups) {
                const uint4 x = *reinterpret_cast<const uint4*>(src + w * rstride);
                const uint64_t d = G == 1 ? dsh : dw2[w], kv = kv2[w];
                uint4 y;
                if constexpr (ES == 2) {
                    y.x = P::narrow(ffma2(kv, dp[0], fmul2(P::widen(x.x), d)));
                    y.y = P::narrow(ffma2(kv, dp[1], fmul2(P::widen(x.y), d)));
                    y.z = P::narrow(ffma2(kv, dp[2], fmul2(P::widen(x.z), d)));
                    y.w = P::narrow(ffma2(kv, dp[3], fmul2(P::widen(x.w), d)));
                } else {
                    const uint64_t y0 = ffma2(kv, dp[0], fmul2(((uint64_t)x.y << 32) | x.x, d));
                    const uint64_t y1 = ffma2(kv, dp[PP - 1], fmul2(((uint64_t)x.w << 32) | x.z, d));
                    y = make_uint4((uint32_t)y0, (uint32_t)(y0 >> 32), (uint32_t)y1, (uint32_t)(y1 >> 32));
                }
                *reinterpret_cast<uint4*>(dst + koff[w]) = y;
            }
        }
        if (more) cp_async_wait_all();  // the next token's slots have landed
        __syncthreads();

        // 3. the read rows, after the write; the next token's write rows are warmed in L2 meanwhile
        ldgsts_rows<E>(rows, bank, qoff, R, sw, row_bytes);
        if (more) {
            const I* rk = reinterpret_cast<const I*>(smem + L.raw_k);
            const int lines = (int)((row_bytes + 127) >> 7);
            const int64_t rowb = (int64_t)hd * ES, colb = (int64_t)c0 * ES;
            for (int i = tid; i < W * lines; i += blockDim.x) {
                const int r = i / lines, l = i - r * lines;
                const unsigned char* p = bank + (int64_t)rk[r] * rowb + colb + (int64_t)l * 128;
                pf_l2(p);
            }
        }
        cp_async_wait_all();
        __syncthreads();
        if (active) {
            uint64_t acc = 0;
            int r = 0;
            if constexpr (sizeof(E) == 2) {
                // bf16 rows: the rounded read weight and the row element are both bf16, so the
                // mixed-precision fma (bf16 operands, float32 accumulator, one rounding) gives the
                // same float32 as widening both and using fmaf
                float lo = 0.0f, hi = 0.0f;
                for (; r + 4 <= R; r += 4) {
                    const uint32_t x0 = rp[(r + 0) * pstride], x1 = rp[(r + 1) * pstride];
                    const uint32_t x2 = rp[(r + 2) * pstride], x3 = rp[(r + 3) * pstride];
                    const uint4 q = *reinterpret_cast<const uint4*>(qv2 + r);  // low words: float32 bits
                    const uint4 q2 = *reinterpret_cast<const uint4*>(qv2 + r + 2);
                    fma_bf16_pair(lo, hi, q.x, x0);
                    fma_bf16_pair(lo, hi, q.z, x1);
                    fma_bf16_pair(lo, hi, q2.x, x2);
                    fma_bf16_pair(lo, hi, q2.z, x3);
                }
                for (; r < R; ++r) fma_bf16_pair(lo, hi, (uint32_t)qv2[r], rp[r * pstride]);
                acc = f2(lo, hi);
            } else {
                for (; r + 4 <= R; r += 4) {
                    const PT x0 = rp[(r + 0) * pstride], x1 = rp[(r + 1) * pstride];
                    const PT x2 = rp[(r + 2) * pstride], x3 = rp[(r + 3) * pstride];
                    const ulonglong2 q01 = *reinterpret_cast<const ulonglong2*>(qv2 + r);
                    const ulonglong2 q23 = *reinterpret_cast<const ulonglong2*>(qv2 + r + 2);
                    acc = ffma2(q01.x, P::widen(x0), acc);
                    acc = ffma2(q01.y, P::widen(x1), acc);
                    acc = ffma2(q23.x, P::widen(x2), acc);
                    acc = ffma2(q23.y, P::widen(x3), acc);
                }
                for (; r < R; ++r) acc = ffma2(qv2[r], P::widen(rp[r * pstride]), acc);
            }
            *reinterpret_cast<PT*>(out + ts * hd + c0 + j) = P::narrow(acc);
        }

        // 4. the next token's metadata (rows and metadata of this token are no longer read)
        cp_async_wait_all();
        __syncthreads();
        if (t + 1 < a.T) derive_meta<E, I>(a, c0, L, smem);
        __syncthreads();
    }
}


// acc + q * x with q the bf16 in the high half of the float32 pattern qbits and x a bf16 element
__device__ __forceinline__ float fma_bf16(float acc, uint32_t qbits, uint16_t x) {
    asm("{\n\t.reg .b16 ql, qh;\n\tmov.b32 {ql, qh}, %1;\n\tfma.rn.f32.bf16 %0, qh, %2, %0;\n\t}"
        : "+f"(acc)
        : "r"(qbits), "h"(x));
    return acc;
}

// the row of entry i of a flattened (row, 128-byte line) list: a shift when the lines per row are a
// power of two (lsh >= 0), else a division (the few-stream kernel below measured 4 % faster per
// launch without the division)
__device__ __forceinline__ int line_row(int i, int lines, int lsh) { return lsh >= 0 ? i >> lsh : i / lines; }

// The staged path for bf16 slices of up to 64 columns with one column per thread: the same
// staging, order of operations and write-back as decode_vec_kernel, scalar chains (each lane of a
// paired op is an independent round-to-nearest op, so the bits are the same) and twice the warps.
template <typename I, bool PIECE, int SW = 0>
__global__ void __launch_bounds__(128, 7) decode_vec1_kernel(const DecodeArgs a, int early_trigger) {
    using E = uint16_t;
    using P = Pair<E>;
    constexpr int ES = 2;
    extern __shared__ __align__(128) unsigned char smem[];

    const int W = a.W, R = a.R, G = a.G, hd = a.hd, sw = SW ? SW : a.slice_cols;
    const VecLayout L(W, R, G, sw, ES, (int)sizeof(I));
    E* rows = reinterpret_cast<E*>(smem + L.rows);
    const int64_t* koff = reinterpret_cast<const int64_t*>(smem + L.koff);
    const int64_t* qoff = reinterpret_cast<const int64_t*>(smem + L.qoff);
    const uint64_t* aw2 = reinterpret_cast<const uint64_t*>(smem + L.aw2);
    const uint64_t* kv2 = reinterpret_cast<const uint64_t*>(smem + L.kv2);
    const uint64_t* dw2 = reinterpret_cast<const uint64_t*>(smem + L.dw2);
    const uint64_t* qv2 = reinterpret_cast<const uint64_t*>(smem + L.qv2);

    const int tid = threadIdx.x, nt = blockDim.x;
    const int64_t s = blockIdx.x / a.n_slices;
    const int c0 = (int)(blockIdx.x % a.n_slices) * sw;
    const int ncols = min(sw, hd - c0);
    const int j = tid;
    const bool active = j < ncols;
    const uint32_t row_bytes = (uint32_t)ncols * ES;
    unsigned char* bank = static_cast<unsigned char*>(a.bank);
    E* out = static_cast<E*>(a.out);
    const E* rc = rows + tid;  // this thread's element of row 0
    const int64_t jb = (int64_t)j * ES;
    const int cpr = (int)(row_bytes >> 4);
    const bool by_piece = PIECE && a.piece_write && nt % cpr == 0 && nt / cpr <= W;
    const int lines = (int)((row_bytes + 127) >> 7);  // 128-byte lines per row slice
    const int lsh = (lines & (lines - 1)) == 0 ? 31 - __clz(lines) : -1;

    // With inputs_ready the inputs predate the preceding kernel: token 0's metadata is read and its
    // rows are warmed in L2 before waiting for that kernel; the bank is read and written (and `out`
    // written) only after the wait. L2 is the point of coherence, so a line warmed early still
    // holds every later write to it. The next launch is released only after the wait, so at most
    // one launch runs its early part ahead of the kernel that is working.
    if (!a.inputs_ready) {
        grid_dependency_wait();
        if (early_trigger) grid_launch_dependents();
    }
    prefetch_meta<I>(a, s * a.sstride, L, smem);  // token 0
    cp_async_wait_all();
    __syncthreads();
    if (G == 1 && tid == 0)
        *reinterpret_cast<float*>(smem + L.dnext) = gate(*reinterpret_cast<const float*>(smem + L.raw_g));
    __syncthreads();
    derive_meta<E, I>(a, c0, L, smem);
    __syncthreads();
    if (a.inputs_ready) {
        prefetch_rows_l2(bank, koff, W, row_bytes);
        prefetch_rows_l2(bank, qoff, R, row_bytes);
        grid_dependency_wait();
        if (early_trigger) grid_launch_dependents();
    }

    for (int t = 0; t < a.T; ++t) {
        const int64_t ts = (int64_t)t * a.tstride + s * a.sstride;

        ldgsts_rows<E>(rows, bank, koff, W, sw, row_bytes);
        for (int i = tid; i < R * lines; i += nt) {
            const int r = line_row(i, lines, lsh), l = i - r * lines;
            pf_l2(bank + qoff[r] + (int64_t)l * 128);
        }
        const float vr = active ? round_to<E>(__ldg(a.v + ts * hd + c0 + j)) : 0.0f;
        const float beta = *reinterpret_cast<const float*>(smem + L.beta);
        const float dsh = f2lo(dw2[0]);
        const bool more = t + 1 < a.T;
        if (more) {
            prefetch_meta<I>(a, ts + a.tstride, L, smem);
            if (G == 1 && tid == 0)
                *reinterpret_cast<float*>(smem + L.dnext) = gate(__ldg(a.g + ts + a.tstride));
        }
        if (more)
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        else
            cp_async_wait_all();
        __syncthreads();

        if (active) {
            float acc = 0.0f;
            int w = 0;
#pragma unroll 4  // 16 rows' loads ahead of their fmas (32-row steps: 6 % faster than the default)
            for (; w + 4 <= W; w += 4) {
                const E x0 = rc[(w + 0) * sw], x1 = rc[(w + 1) * sw], x2 = rc[(w + 2) * sw], x3 = rc[(w + 3) * sw];
                const ulonglong2 a01 = *reinterpret_cast<const ulonglong2*>(aw2 + w);
                const ulonglong2 a23 = *reinterpret_cast<const ulonglong2*>(aw2 + w + 2);
                acc = fmaf(f2lo(a01.x), to_f32(x0), acc);
                acc = fmaf(f2lo(a01.y), to_f32(x1), acc);
                acc = fmaf(f2lo(a23.x), to_f32(x2), acc);
                acc = fmaf(f2lo(a23.y), to_f32(x3), acc);
            }
            for (; w < W; ++w) acc = fmaf(f2lo(aw2[w]), to_f32(rc[w * sw]), acc);
            const float delta = __fmul_rn(beta, __fsub_rn(vr, acc));
            if (by_piece) {
                reinterpret_cast<float*>(smem + L.dlt)[tid] = delta;
            } else {
                unsigned char* bj = bank + jb;
                for (w = 0; w < W; ++w) {
                    const float y = fmaf(f2lo(kv2[w]), delta, __fmul_rn(to_f32(rc[w * sw]), G == 1 ? dsh : f2lo(dw2[w])));
                    *reinterpret_cast<E*>(bj + koff[w]) = from_f32<E>(y);
                }
            }
        }
        if (by_piece) {
            __syncthreads();
            constexpr int PP = 16 / (2 * ES);
            const int k = tid % cpr, ngroups = nt / cpr;
            const uint64_t d_sh = dw2[0];
            uint64_t dp[PP];
#pragma unroll
            for (int p = 0; p < PP; ++p) dp[p] = reinterpret_cast<const uint64_t*>(smem + L.dlt)[k * PP + p];
            const unsigned char* src = reinterpret_cast<const unsigned char*>(rows) + k * 16;
            unsigned char* dst = bank + k * 16;
            const size_t rstride = (size_t)sw * ES;
#pragma unroll 2
            for (int w = tid / cpr; w < W; w += ngroups) {
                const uint4 x = *reinterpret_cast<const uint4*>(src + w * rstride);
                const uint64_t d = G == 1 ? d_sh : dw2[w], kv = kv2[w];
                uint4 y;
                y.x = P::narrow(ffma2(kv, dp[0], fmul2(P::widen(x.x), d)));
                y.y = P::narrow(ffma2(kv, dp[1], fmul2(P::widen(x.y), d)));
                y.z = P::narrow(ffma2(kv, dp[2], fmul2(P::widen(x.z), d)));
                y.w = P::narrow(ffma2(kv, dp[3], fmul2(P::widen(x.w), d)));
                *reinterpret_cast<uint4*>(dst + koff[w]) = y;
            }
        }
        if (more) cp_async_wait_all();
        __syncthreads();

        ldgsts_rows<E>(rows, bank, qoff, R, sw, row_bytes);
        if (more) {
            const I* rk = reinterpret_cast<const I*>(smem + L.raw_k);
            const int64_t rowb = (int64_t)hd * ES, colb = (int64_t)c0 * ES;
            for (int i = tid; i < W * lines; i += nt) {
                const int r = line_row(i, lines, lsh), l = i - r * lines;
                const unsigned char* p = bank + (int64_t)rk[r] * rowb + colb + (int64_t)l * 128;
                pf_l2(p);
            }
        }
        cp_async_wait_all();
        __syncthreads();
        if (active) {
            float acc = 0.0f;
            int r = 0;
#pragma unroll 4
            for (; r + 4 <= R; r += 4) {
                const uint4 q = *reinterpret_cast<const uint4*>(qv2 + r);
                const uint4 q2 = *reinterpret_cast<const uint4*>(qv2 + r + 2);
                acc = fma_bf16(acc, q.x, rc[(r + 0) * sw]);
                acc = fma_bf16(acc, q.z, rc[(r + 1) * sw]);
                acc = fma_bf16(acc, q2.x, rc[(r + 2) * sw]);
                acc = fma_bf16(acc, q2.z, rc[(r + 3) * sw]);
            }
            for (; r < R; ++r) acc = fma_bf16(acc, (uint32_t)qv2[r], rc[r * sw]);
            out[ts * hd + c0 + j] = from_f32<E>(acc);
        }

        cp_async_wait_all();
        __syncthreads();
        if (t + 1 < a.T) derive_meta<E, I>(a, c0, L, smem);
        __syncthreads();
    }
}

// ---------------------------------------------------------------- streaming path (wide rows)
// When W or R rows do not fit the shared-memory budget at a useful slice width (e.g. 256 rows of
// 1 KiB), the rows stream through a ring of NS chunk buffers of CH rows each instead of being
// staged all at once: the write rows pass twice (retrieve, then decay-and-write; the second pass
// is served mostly by L2) and the read rows once. Chunks are consumed in ascending row order, so
// every sum keeps the order and the bits of the staged path. NS and CH are chosen at launch: CH
// is the largest chunk (kStreamRowsMin..kStreamRowsMax rows) whose ring still lets every block of
// the grid be resident at once (larger chunks put more rows in flight and take fewer barriers per
// pass), with NS = 3 when that allows chunks of kTallChunk rows or more, else NS = 4.

constexpr int kStreamRowsMin = 16;  // rows per chunk, at least
constexpr int kStreamRowsMax = 32;  // and at most
constexpr int kTallChunk = 24;      // three stages suffice from this chunk height on

struct StreamLayout {
    VecLayout meta;  // the metadata of the staged layout, with no row area
    size_t ring, total;
    __host__ __device__ StreamLayout(int W, int R, int G, int sw, int es, int is, int ch, int ns)
        : meta(W, R, G, 0, es, is) {
        ring = align_up(meta.total, 128);
        total = ring + (size_t)ns * ch * sw * es;
    }
};

// Every thread: rows [r0, r0 + n) of off[] into ring buffer dst; one commit group.
template <typename E>
__device__ __forceinline__ void ldgsts_chunk(unsigned char* dst, const unsigned char* bank, const int64_t* off, int r0,
                                             int n, int sw, uint32_t row_bytes) {
    ldgsts_rows<E>(reinterpret_cast<E*>(dst), bank, off + r0, n, sw, row_bytes);
}

template <typename E, typename I, int NS>
__global__ void __launch_bounds__(kMaxThreads, 1) decode_stream_kernel(const DecodeArgs a, int early_trigger) {
    using P = Pair<E>;
    using PT = typename P::T;
    constexpr int ES = sizeof(E);
    const int CH = a.stream_rows;
    extern __shared__ __align__(128) unsigned char smem[];

    const int W = a.W, R = a.R, G = a.G, hd = a.hd, sw = a.slice_cols;
    const StreamLayout SL(W, R, G, sw, ES, (int)sizeof(I), CH, NS);
    const VecLayout& L = SL.meta;
    unsigned char* ring = smem + SL.ring;
    const size_t stage_bytes = (size_t)CH * sw * ES;
    const int64_t* koff = reinterpret_cast<const int64_t*>(smem + L.koff);
    const int64_t* qoff = reinterpret_cast<const int64_t*>(smem + L.qoff);
    const uint64_t* aw2 = reinterpret_cast<const uint64_t*>(smem + L.aw2);
    const uint64_t* kv2 = reinterpret_cast<const uint64_t*>(smem + L.kv2);
    const uint64_t* dw2 = reinterpret_cast<const uint64_t*>(smem + L.dw2);
    const uint64_t* qv2 = reinterpret_cast<const uint64_t*>(smem + L.qv2);

    const int tid = threadIdx.x;
    const int64_t s = blockIdx.x / a.n_slices;
    const int c0 = (int)(blockIdx.x % a.n_slices) * sw;
    const int ncols = min(sw, hd - c0);
    const int j = 2 * tid;
    const bool active = j < ncols;
    const uint32_t row_bytes = (uint32_t)ncols * ES;
    const int pstride = sw / 2;
    unsigned char* bank = static_cast<unsigned char*>(a.bank);
    E* out = static_cast<E*>(a.out);
    const int64_t jb = (int64_t)j * ES;
    const int nk = (W + CH - 1) / CH, nq = (R + CH - 1) / CH;
    // row pair of this thread in row r of ring stage st
    const auto at = [&](int st, int r) -> PT {
        return reinterpret_cast<const PT*>(ring + st * stage_bytes)[r * pstride + tid];
    };

    // With inputs_ready the inputs predate the preceding kernel: token 0's metadata is read and its
    // rows are warmed in L2 before waiting for that kernel; the bank is read and written (and `out`
    // written) only after the wait. L2 is the point of coherence, so a line warmed early still
    // holds every later write to it. The next launch is released only after the wait, so at most
    // one launch runs its early part ahead of the kernel that is working.
    if (!a.inputs_ready) {
        grid_dependency_wait();
        if (early_trigger) grid_launch_dependents();
    }
    prefetch_meta<I>(a, s * a.sstride, L, smem);  // token 0
    cp_async_wait_all();
    __syncthreads();
    if (G == 1 && tid == 0)
        *reinterpret_cast<float*>(smem + L.dnext) = gate(*reinterpret_cast<const float*>(smem + L.raw_g));
    __syncthreads();
    derive_meta<E, I>(a, c0, L, smem);
    __syncthreads();
    if (a.inputs_ready) {
        prefetch_rows_l2(bank, koff, W, row_bytes);
        prefetch_rows_l2(bank, qoff, R, row_bytes);
        grid_dependency_wait();
        if (early_trigger) grid_launch_dependents();
    }

    for (int t = 0; t < a.T; ++t) {
        const int64_t ts = (int64_t)t * a.tstride + s * a.sstride;
        uint64_t vr = 0;
        if (active) {
            const float2 vv = __ldg(reinterpret_cast<const float2*>(a.v + ts * hd + c0 + j));
            vr = P::widen(P::narrow(f2(vv.x, vv.y)));
        }
        const float beta = *reinterpret_cast<const float*>(smem + L.beta);
        const uint64_t dsh = dw2[0];

        // passes 1 and 2: job q < nk retrieves over write chunk q; job q >= nk writes chunk q - nk
        uint64_t acc = 0, delta = 0;
        const int jobs = 2 * nk;
        // exactly NS - 1 groups ahead (empty ones past the last job), so that after job q's own
        // group the wait for "at most NS - 1 pending" always covers job q
        for (int q = 0; q < NS - 1; ++q) {
            if (q < jobs) {
                const int c = q % nk;
                ldgsts_chunk<E>(ring + (q % NS) * stage_bytes, bank, koff, c * CH, min(CH, W - c * CH), sw, row_bytes);
            } else {
                cp_async_commit();
            }
        }
        for (int q = 0; q < jobs; ++q) {
            const int qn = q + NS - 1;
            if (qn < jobs) {
                const int c = qn % nk;
                ldgsts_chunk<E>(ring + (qn % NS) * stage_bytes, bank, koff, c * CH, min(CH, W - c * CH), sw, row_bytes);
            } else {
                cp_async_commit();  // keep one group per job
            }
            asm volatile("cp.async.wait_group %0;" ::"n"(NS - 1) : "memory");
            __syncthreads();
            const int st = q % NS, c = q % nk, r0 = c * CH, n = min(CH, W - r0);
            if (active) {
                if (q < nk) {
                    for (int r = 0; r < n; ++r) acc = ffma2(aw2[r0 + r], P::widen(at(st, r)), acc);
                } else {
                    if (q == nk) {
                        const float dl = __fmul_rn(beta, __fsub_rn(f2lo(vr), f2lo(acc)));
                        const float dh = __fmul_rn(beta, __fsub_rn(f2hi(vr), f2hi(acc)));
                        delta = f2(dl, dh);
                    }
                    for (int r = 0; r < n; ++r) {
                        const int w = r0 + r;
                        const uint64_t y = ffma2(kv2[w], delta, fmul2(P::widen(at(st, r)), G == 1 ? dsh : dw2[w]));
                        *reinterpret_cast<PT*>(bank + koff[w] + jb) = P::narrow(y);
                    }
                }
            }
            __syncthreads();  // stage st is refilled by the next iteration's copy
        }

        // pass 3: the read rows, after every write of this token; the next token's metadata too
        const bool more = t + 1 < a.T;
        if (more) {
            prefetch_meta<I>(a, ts + a.tstride, L, smem);
            if (G == 1 && tid == 0)
                *reinterpret_cast<float*>(smem + L.dnext) = gate(__ldg(a.g + ts + a.tstride));
        }
        uint64_t racc = 0;
        for (int q = 0; q < NS - 1; ++q) {
            if (q < nq)
                ldgsts_chunk<E>(ring + (q % NS) * stage_bytes, bank, qoff, q * CH, min(CH, R - q * CH), sw, row_bytes);
            else
                cp_async_commit();
        }
        for (int q = 0; q < nq; ++q) {
            const int qn = q + NS - 1;
            if (qn < nq)
                ldgsts_chunk<E>(ring + (qn % NS) * stage_bytes, bank, qoff, qn * CH, min(CH, R - qn * CH), sw, row_bytes);
            else
                cp_async_commit();
            asm volatile("cp.async.wait_group %0;" ::"n"(NS - 1) : "memory");
            __syncthreads();
            const int st = q % NS, r0 = q * CH, n = min(CH, R - r0);
            if (active)
                for (int r = 0; r < n; ++r) racc = ffma2(qv2[r0 + r], P::widen(at(st, r)), racc);
            __syncthreads();
        }
        if (active) *reinterpret_cast<PT*>(out + ts * hd + c0 + j) = P::narrow(racc);

        // the next token's metadata
        cp_async_wait_all();
        __syncthreads();
        if (more) derive_meta<E, I>(a, c0, L, smem);
        __syncthreads();
    }
}

// ---------------------------------------------------------------- streaming path, float32, a column per thread
//
// Float32 banks whose W or R rows cannot all be staged (e.g. 256 rows of 1 KiB) stream their row
// slices through a ring of NS chunks of CH rows, one column per thread, slices of up to 256
// columns chosen at launch so that the grid balances over the SMs (e.g. 256 streams of 1 KiB rows:
// 1024 quarter-row blocks, 7 per SM). The block's metadata is kept lean so that the ring stays
// deep at that occupancy: the slots as row indices, 32-bit wherever a slot cannot reach 2^32 (int32
// slots; int64 slots of rows of at least 64 columns, where 2^32 rows would make a bank of over 1 TiB)
// and single float weights.
//
// Each block runs one job list per "segment": the read chunks of token t-1, then the retrieve
// chunks and the decay-and-write chunks of token t (the write rows pass twice: retrieve, then
// write; the second pass is served by L2). The ring runs through a segment without draining: the
// read rows of token t-1 and the write rows of token t are both read after token t-1's writes and
// before token t's, so their copies can run back to back. It drains only at the end of a segment,
// where token t's writes must be complete before token t's read rows are copied. A chunk's stage
// is refilled as soon as every thread has consumed it, before the next chunk is awaited, so that
// all NS stages are in flight during each wait. The launcher uses two stages of chunks as tall as
// the shared memory allows (up to kWideRowsMax rows): every chunk costs two barriers and a wait,
// and fewer, taller chunks measured faster than more stages of shorter ones (256 streams: two
// stages of 48 rows 0.285 ms, three of 32 0.293 ms, four of 24 0.327 ms).
// Chunks are consumed in ascending row order, so every sum keeps the staged path's order and bits.
// The decay-and-write stores 16-byte pieces (four columns of a row) rather than a column per thread,
// from the column deltas that the retrieve's last job publishes in shared memory (1 % faster on the
// 256-stream workload). The readings and the written-back rows are stored evict-first in L2: what
// L2 should keep are the write rows between their two passes and the rows warmed for the next
// copies.

// sb: bytes per stored slot (4 or 8)
struct WideLayout {
    size_t koff, kv, dw, beta, qoff, qv, dlt, ring, total;
    __host__ __device__ WideLayout(int W, int R, int G, int sw, int ch, int ns, int sb) {
        koff = 0;  // the write side: slots, weights, log-decays turned into gates in place
        kv = align_up(koff + (size_t)W * sb, 16);
        dw = align_up(kv + (size_t)W * 4, 16);
        beta = align_up(dw + (size_t)G * 4, 16);
        qoff = align_up(beta + 4, 16);  // the read side: slots, weights
        qv = align_up(qoff + (size_t)R * sb, 16);
        dlt = align_up(qv + (size_t)R * 4, 16);  // the slice's deltas, read by the write-back's pieces
        ring = align_up(dlt + (size_t)sw * 4, 128);
        total = ring + (size_t)ns * ch * sw * 4;
    }
};

// a slot copied into S (32-bit for a 64-bit slot below 2^32: its low word, little-endian)
template <typename S>
__device__ __forceinline__ void cp_async_slot(S* dst, const void* src) {
    if constexpr (sizeof(S) == 8)
        cp_async8(dst, src);
    else
        cp_async4(dst, src);
}

// Every thread: cp.async copies of token ts's write-side inputs in place: the slots into the slot
// array, the weights into kv, the log-decays into dw, beta (no commit). wide_derive_k turns the
// log-decays into gates.
template <typename I, typename S>
__device__ __forceinline__ void wide_load_k(const DecodeArgs& a, int64_t ts, const WideLayout& L, unsigned char* smem) {
    const int tid = threadIdx.x, nt = blockDim.x, W = a.W, G = a.G;
    S* rk = reinterpret_cast<S*>(smem + L.koff);
    float* kv = reinterpret_cast<float*>(smem + L.kv);
    float* dw = reinterpret_cast<float*>(smem + L.dw);
    const I* k_idx = static_cast<const I*>(a.k_idx) + ts * W;
    for (int i = tid; i < W; i += nt) {
        cp_async_slot(rk + i, k_idx + i);
        cp_async4(kv + i, a.k_val + ts * W + i);
    }
    for (int i = tid; i < G; i += nt) cp_async4(dw + i, a.g + ts * G + i);
    if (tid == 0) cp_async4(smem + L.beta, a.beta + ts);
}

// Every thread: cp.async copies of token ts's read-side inputs: the slots into the slot array, the
// weights into qv (no commit). They are used as copied.
template <typename I, typename S>
__device__ __forceinline__ void wide_load_q(const DecodeArgs& a, int64_t ts, const WideLayout& L, unsigned char* smem) {
    const int tid = threadIdx.x, nt = blockDim.x, R = a.R;
    S* rq = reinterpret_cast<S*>(smem + L.qoff);
    float* qv = reinterpret_cast<float*>(smem + L.qv);
    const I* q_idx = static_cast<const I*>(a.q_idx) + ts * R;
    for (int i = tid; i < R; i += nt) {
        cp_async_slot(rq + i, q_idx + i);
        cp_async4(qv + i, a.q_val + ts * R + i);
    }
}

// Every thread: the write side's log-decays become gates d = exp(g) in place, each by the thread
// that copied it (a shared gate by thread 0); the weights are used as given (a = kv * d is formed
// where it is used).
__device__ __forceinline__ void wide_derive_k(const DecodeArgs& a, const WideLayout& L, unsigned char* smem) {
    float* dw = reinterpret_cast<float*>(smem + L.dw);
    if (a.G == 1) {
        if (threadIdx.x == 0) dw[0] = gate(dw[0]);
    } else {
        for (int i = threadIdx.x; i < a.G; i += blockDim.x) dw[i] = gate(dw[i]);
    }
}

// Every thread: 16-byte cp.async copies of n row slices, row slot[r] of the bank at base (the slice's
// first column), into rows[r * sw]; one commit group.
template <typename S>
__device__ __forceinline__ void ldgsts_slots(float* rows, const unsigned char* base, const S* slot, int n, int sw,
                                             uint32_t row_bytes, uint32_t rowb) {
    const int tid = threadIdx.x, nt = blockDim.x;
    const int cpr = (int)(row_bytes >> 4);  // 16-byte chunks per row slice
    unsigned char* dst = reinterpret_cast<unsigned char*>(rows);
    const size_t rs = (size_t)sw * 4;
    if (nt % cpr == 0) {
        const int k = tid % cpr, step = nt / cpr;
        for (int r = tid / cpr; r < n; r += step)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst + r * rs + k * 16)),
                         "l"(base + (uint64_t)slot[r] * rowb + k * 16)
                         : "memory");
    } else {
        for (int c = tid; c < n * cpr; c += nt) {
            const int r = c / cpr, k = c - r * cpr;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst + r * rs + k * 16)),
                         "l"(base + (uint64_t)slot[r] * rowb + k * 16)
                         : "memory");
        }
    }
    cp_async_commit();
}

constexpr int kWideRegs = 128;  // registers per thread of decode_wide_kernel, at most (2 blocks of 256)

// S: the stored slot type (uint32_t, or int64_t for 64-bit slots that may reach 2^32)
template <typename I, int NS, int SW = 0, typename S = uint32_t>
__global__ void __launch_bounds__(kMaxThreads, 65536 / (kMaxThreads * kWideRegs))
    decode_wide_kernel(const DecodeArgs a, int early_trigger) {
    const int CH = a.stream_rows;
    extern __shared__ __align__(128) unsigned char smem[];

    const int W = a.W, R = a.R, G = a.G, hd = a.hd, sw = SW ? SW : a.slice_cols, T = a.T;
    const WideLayout L(W, R, G, sw, CH, NS, sizeof(S));
    unsigned char* ring = smem + L.ring;
    const size_t stage_bytes = (size_t)CH * sw * 4;
    const S* kslot = reinterpret_cast<const S*>(smem + L.koff);
    const S* qslot = reinterpret_cast<const S*>(smem + L.qoff);
    const float* kv = reinterpret_cast<const float*>(smem + L.kv);
    const float* dw = reinterpret_cast<const float*>(smem + L.dw);
    const float* qv = reinterpret_cast<const float*>(smem + L.qv);

    const int tid = threadIdx.x;  // this thread's column within the slice
    float* out = static_cast<float*>(a.out);
    const int64_t jb = (int64_t)tid * 4;
    const int nk = (W + CH - 1) / CH, nq = (R + CH - 1) / CH;
    const int64_t s = blockIdx.x / a.n_slices;
    const int c0 = (int)(blockIdx.x % a.n_slices) * sw;
    // row slot w of the slice: base + slot * rowb
    unsigned char* base = static_cast<unsigned char*>(a.bank) + (int64_t)c0 * 4;
    const uint32_t rowb = (uint32_t)hd * 4;
    const int ncols = min(sw, hd - c0);
    const bool active = tid < ncols;
    const uint32_t row_bytes = (uint32_t)ncols * 4;
    const int nt = blockDim.x, cpr = (int)(row_bytes >> 4);  // 16-byte pieces per row slice
    const bool by_piece = nt % cpr == 0;  // the write-back by pieces (else a column per thread)

    // With inputs_ready the inputs predate the preceding kernel: token 0's write side is read and its
    // rows are warmed in L2 before waiting for that kernel; the bank is read and written (and `out`
    // written) only after the wait.
    if (!a.inputs_ready) {
        grid_dependency_wait();
        if (early_trigger) grid_launch_dependents();
    }
    const int64_t ts0 = s * a.sstride;  // token 0 of this stream
    wide_load_k<I, S>(a, ts0, L, smem);
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    wide_derive_k(a, L, smem);
    __syncthreads();
    // the write side of a later token is copied at the start of its segment and derived before its
    // first write-row copy, which the ring issues NS - 1 jobs ahead: at job nq - NS + 1
    const int kd = nq - NS + 1;
    if (a.inputs_ready) {
        const int lines = (int)((row_bytes + 127) >> 7);
        for (int i = tid; i < W * lines; i += blockDim.x) {
            const int r = i / lines, l = i - r * lines;
            pf_l2(base + (uint64_t)kslot[r] * rowb + l * 128);
        }
        grid_dependency_wait();
        if (early_trigger) grid_launch_dependents();
    }

    float racc = 0.0f, acc = 0.0f, delta = 0.0f, vr = 0.0f, beta = 0.0f, d1 = 1.0f;
    for (int t = 0; t <= T; ++t) {
        const int nr = t > 0 ? nq : 0;       // read chunks of token t-1
        const int nkk = t < T ? 2 * nk : 0;  // retrieve and write chunks of token t
        const int jobs = nr + nkk;
        const int64_t tsk = ts0 + (int64_t)t * a.tstride;  // token t's row of the inputs
        if (t > 0) {
            // token t-1's writes are done (every thread passed its last job before this barrier), so
            // the write side is free for token t's, and token t-1's read side has landed
            cp_async_wait_all();
            __syncthreads();
            if (t < T) {
                wide_load_k<I, S>(a, tsk, L, smem);
                cp_async_commit();  // the oldest group: landed once job 0 has
                if (kd < 1) {       // few read chunks: the first write-row copy is in the ring's prologue
                    cp_async_wait_all();
                    __syncthreads();
                    wide_derive_k(a, L, smem);
                    __syncthreads();
                }
            }
        }
        const bool k_ready = t == 0 || kd < 1;  // token t's write side derived before the jobs
        const auto load_token_state = [&]() {
            if (active) vr = __ldg(a.v + tsk * hd + c0 + tid);
            beta = *reinterpret_cast<const float*>(smem + L.beta);
            d1 = dw[0];
            acc = 0.0f;
        };
        if (t < T && k_ready) load_token_state();
        const auto issue = [&](int q) {
            if (q < jobs) {
                unsigned char* dst = ring + (q % NS) * stage_bytes;
                if (q < nr) {
                    const int r0 = q * CH;
                    ldgsts_slots(reinterpret_cast<float*>(dst), base, qslot + r0, min(CH, R - r0), sw, row_bytes, rowb);
                } else {
                    const int r0 = ((q - nr) % nk) * CH;
                    ldgsts_slots(reinterpret_cast<float*>(dst), base, kslot + r0, min(CH, W - r0), sw, row_bytes, rowb);
                }
            } else {
                cp_async_commit();  // one group per job, so that the waits below count jobs
            }
        };
        for (int q = 0; q < NS - 1; ++q) issue(q);
        // Once token t-1's read rows are all consumed (the first job after them), token t's read side
        // is copied in place; its commit group then sits among the ring's.
        const int meta_job = t < T ? nr : -1;
        for (int q = 0; q < jobs; ++q) {
            if (t < T && !k_ready && q == kd) {  // token t's write side has landed (job 0 waited for it)
                wide_derive_k(a, L, smem);
                __syncthreads();
                load_token_state();
            }
            // refill the stage that job q-1 used (every thread is done with it: the barrier that
            // ends job q-1), so that all NS stages are in flight while job q is awaited
            issue(q + NS - 1);
            if (q == meta_job) {
                wide_load_q<I, S>(a, tsk, L, smem);
                cp_async_commit();
            }
            // job q has landed: at most NS - 1 younger groups pending, one more while the metadata
            // group committed after job q's is among them
            if (meta_job >= 0 && q >= meta_job && q <= meta_job + NS - 1)
                asm volatile("cp.async.wait_group %0;" ::"n"(NS) : "memory");
            else
                asm volatile("cp.async.wait_group %0;" ::"n"(NS - 1) : "memory");
            __syncthreads();  // job q is visible to every thread
            // this thread's column of the chunk's rows; chunk heights are a multiple of 4, so the
            // per-row metadata of four rows is one 16-byte load
            const float* x = reinterpret_cast<const float*>(ring + (q % NS) * stage_bytes) + tid;
            if (q < nr) {  // readings of token t-1
                const int r0 = q * CH, n = min(CH, R - r0);
                if (active) {
                    int r = 0;
                    for (; r + 4 <= n; r += 4) {
                        const float4 q4 = *reinterpret_cast<const float4*>(qv + r0 + r);
                        racc = fmaf(q4.x, x[(r + 0) * sw], racc);
                        racc = fmaf(q4.y, x[(r + 1) * sw], racc);
                        racc = fmaf(q4.z, x[(r + 2) * sw], racc);
                        racc = fmaf(q4.w, x[(r + 3) * sw], racc);
                    }
                    for (; r < n; ++r) racc = fmaf(qv[r0 + r], x[r * sw], racc);
                    if (q == nr - 1) {
                        st_hint(out + (tsk - a.tstride) * hd + c0 + tid, racc, l2_evict_first());
                        racc = 0.0f;
                    }
                }
            } else if (q < nr + nk) {  // retrieve of token t: a_w = kv_w * d_w, then the fma chain
                const int r0 = (q - nr) * CH, n = min(CH, W - r0);
                if (active) {
                    int r = 0;
                    for (; r + 4 <= n; r += 4) {
                        const float4 k4 = *reinterpret_cast<const float4*>(kv + r0 + r);
                        float4 d4 = make_float4(d1, d1, d1, d1);
                        if (G != 1) d4 = *reinterpret_cast<const float4*>(dw + r0 + r);
                        acc = fmaf(__fmul_rn(k4.x, d4.x), x[(r + 0) * sw], acc);
                        acc = fmaf(__fmul_rn(k4.y, d4.y), x[(r + 1) * sw], acc);
                        acc = fmaf(__fmul_rn(k4.z, d4.z), x[(r + 2) * sw], acc);
                        acc = fmaf(__fmul_rn(k4.w, d4.w), x[(r + 3) * sw], acc);
                    }
                    for (; r < n; ++r) {
                        const int w = r0 + r;
                        acc = fmaf(__fmul_rn(kv[w], G == 1 ? d1 : dw[w]), x[r * sw], acc);
                    }
                    if (q == nr + nk - 1)  // the column's delta, published by the barrier that ends this job
                        reinterpret_cast<float*>(smem + L.dlt)[tid] = __fmul_rn(beta, __fsub_rn(vr, acc));
                }
            } else if (by_piece) {  // decay-and-write of token t, one 16-byte piece (4 columns) at a time
                const int r0 = (q - nr - nk) * CH, n = min(CH, W - r0);
                const int k = tid % cpr, ng = nt / cpr;
                const float4 dl = reinterpret_cast<const float4*>(smem + L.dlt)[k];
                const unsigned char* stg = ring + (q % NS) * stage_bytes + k * 16;
                const uint64_t ef = l2_evict_first();
                for (int r = tid / cpr; r < n; r += ng) {
                    const int w = r0 + r;
                    const float4 xv = *reinterpret_cast<const float4*>(stg + (size_t)r * sw * 4);
                    const float kw = kv[w], dd = G == 1 ? d1 : dw[w];
                    st_hint4(base + (uint64_t)kslot[w] * rowb + k * 16, fmaf(kw, dl.x, __fmul_rn(xv.x, dd)),
                             fmaf(kw, dl.y, __fmul_rn(xv.y, dd)), fmaf(kw, dl.z, __fmul_rn(xv.z, dd)),
                             fmaf(kw, dl.w, __fmul_rn(xv.w, dd)), ef);
                }
            } else {  // decay-and-write of token t, this thread's column
                const int r0 = (q - nr - nk) * CH, n = min(CH, W - r0);
                if (active) {
                    if (r0 == 0) delta = __fmul_rn(beta, __fsub_rn(vr, acc));
                    unsigned char* bj = base + jb;
                    int r = 0;
                    for (; r + 4 <= n; r += 4) {
                        const int w = r0 + r;
                        const float4 k4 = *reinterpret_cast<const float4*>(kv + w);
                        float4 d4 = make_float4(d1, d1, d1, d1);
                        if (G != 1) d4 = *reinterpret_cast<const float4*>(dw + w);
                        const uint64_t ef = l2_evict_first();
                        st_hint(reinterpret_cast<float*>(bj + (uint64_t)kslot[w + 0] * rowb), fmaf(k4.x, delta, __fmul_rn(x[(r + 0) * sw], d4.x)), ef);
                        st_hint(reinterpret_cast<float*>(bj + (uint64_t)kslot[w + 1] * rowb), fmaf(k4.y, delta, __fmul_rn(x[(r + 1) * sw], d4.y)), ef);
                        st_hint(reinterpret_cast<float*>(bj + (uint64_t)kslot[w + 2] * rowb), fmaf(k4.z, delta, __fmul_rn(x[(r + 2) * sw], d4.z)), ef);
                        st_hint(reinterpret_cast<float*>(bj + (uint64_t)kslot[w + 3] * rowb), fmaf(k4.w, delta, __fmul_rn(x[(r + 3) * sw], d4.w)), ef);
                    }
                    for (; r < n; ++r) {
                        const int w = r0 + r;
                        st_hint(reinterpret_cast<float*>(bj + (uint64_t)kslot[w] * rowb),
                                fmaf(kv[w], delta, __fmul_rn(x[r * sw], G == 1 ? d1 : dw[w])), l2_evict_first());
                    }
                }
            }
            __syncthreads();  // job q's stage is refilled by the next job's copy
        }
    }
}

// ---------------------------------------------------------------- plain-load path

struct SimtLayout {
    size_t rows, k_slot, q_slot, kv, aw, dw, qv, total;
    __host__ __device__ SimtLayout(int W, int R, int slice_cols, int es) {
        const int maxwr = W > R ? W : R;
        rows = 0;
        k_slot = align_up((size_t)maxwr * slice_cols * es, 16);
        q_slot = k_slot + (size_t)W * 8;
        kv = q_slot + (size_t)R * 8;
        aw = kv + (size_t)W * 4;
        dw = aw + (size_t)W * 4;
        qv = dw + (size_t)W * 4;
        total = qv + (size_t)R * 4;
    }
};

// This thread's column of n rows into rows[i * sw + j].
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

template <typename E, typename I>
__global__ void __launch_bounds__(kMaxThreads) decode_simt_kernel(const DecodeArgs a, int early_trigger) {
    constexpr int ES = sizeof(E);
    extern __shared__ __align__(128) unsigned char smem[];

    const int W = a.W, R = a.R, G = a.G, hd = a.hd, sw = a.slice_cols;
    const SimtLayout L(W, R, sw, ES);
    E* rows = reinterpret_cast<E*>(smem + L.rows);
    int64_t* k_slot = reinterpret_cast<int64_t*>(smem + L.k_slot);
    int64_t* q_slot = reinterpret_cast<int64_t*>(smem + L.q_slot);
    float* kv = reinterpret_cast<float*>(smem + L.kv);
    float* aw = reinterpret_cast<float*>(smem + L.aw);
    float* dw = reinterpret_cast<float*>(smem + L.dw);
    float* qv = reinterpret_cast<float*>(smem + L.qv);

    const int tid = threadIdx.x, nt = blockDim.x;
    const int64_t s = blockIdx.x / a.n_slices;
    const int c0 = (int)(blockIdx.x % a.n_slices) * sw;
    const int ncols = min(sw, hd - c0);
    const int j = tid;
    const bool active = j < ncols;
    E* bank = static_cast<E*>(a.bank);
    E* out = static_cast<E*>(a.out);
    grid_dependency_wait();  // this kernel loads its metadata per token: inputs_ready changes nothing here
    if (early_trigger) grid_launch_dependents();

    for (int t = 0; t < a.T; ++t) {
        const int64_t ts = (int64_t)t * a.tstride + s * a.sstride;
        for (int i = tid; i < W; i += nt) {
            const int64_t e = ts * W + i;
            k_slot[i] = load_index<I>(a.k_idx, e);
            kv[i] = round_to<E>(__ldg(a.k_val + e));
            if (G != 1) dw[i] = gate(__ldg(a.g + ts * G + i));
        }
        if (G == 1 && tid == 0) dw[0] = gate(__ldg(a.g + ts));
        for (int i = tid; i < R; i += nt) {
            const int64_t e = ts * R + i;
            q_slot[i] = load_index<I>(a.q_idx, e);
            qv[i] = round_to<E>(__ldg(a.q_val + e));
        }
        const float vr = active ? round_to<E>(__ldg(a.v + ts * hd + c0 + j)) : 0.0f;
        const float beta = __ldg(a.beta + ts);
        __syncthreads();
        if (active) load_rows_simt<E>(rows, bank, k_slot, W, hd, c0 + j, sw, j);
        for (int i = tid; i < W; i += nt) aw[i] = __fmul_rn(kv[i], dw[G == 1 ? 0 : i]);
        __syncthreads();
        if (active) {
            float acc = 0.0f;
            for (int w = 0; w < W; ++w) acc = fmaf(aw[w], to_f32(rows[(size_t)w * sw + j]), acc);
            const float delta = __fmul_rn(beta, __fsub_rn(vr, acc));
            for (int w = 0; w < W; ++w) {
                const float x = to_f32(rows[(size_t)w * sw + j]);
                bank[k_slot[w] * hd + c0 + j] = from_f32<E>(fmaf(kv[w], delta, __fmul_rn(x, dw[G == 1 ? 0 : w])));
            }
            load_rows_simt<E>(rows, bank, q_slot, R, hd, c0 + j, sw, j);
            acc = 0.0f;
            for (int r = 0; r < R; ++r) acc = fmaf(qv[r], to_f32(rows[(size_t)r * sw + j]), acc);
            out[ts * hd + c0 + j] = from_f32<E>(acc);
        }
        __syncthreads();  // metadata is rewritten by the next token
    }
}

// ---------------------------------------------------------------- launch

enum Path { kSimt = 0, kStaged = 1, kStream = 2 };

// Instances with the slice width fixed at compile time for the common slices: a staged bf16 row
// of 128 columns, a narrow bf16 slice of 64, a streamed float32 quarter row of 64 (measured 1 %
// faster each on the serving and wide workloads, same bits).
template <typename E, typename I, bool PIECE>
auto vec_kernel(int sw) {
    if constexpr (sizeof(E) == 2)
        return sw == 128 ? decode_vec_kernel<E, I, PIECE, 128> : decode_vec_kernel<E, I, PIECE>;
    else
        return decode_vec_kernel<E, I, PIECE>;
}

template <typename I, bool PIECE>
auto vec1_kernel(int sw) {
    return sw == 64 ? decode_vec1_kernel<I, PIECE, 64> : decode_vec1_kernel<I, PIECE>;
}

// bytes per slot that decode_wide_kernel stores: 64-bit slots stay 64-bit only for rows of fewer
// than 64 float32 columns (2^32 rows of 64 columns or more would make a bank of over 1 TiB)
int wide_slot_bytes(int is, int hd) { return is == 8 && hd < 64 ? 8 : 4; }

// the streaming kernel of a bank dtype: float32 banks a column per thread, bf16 banks column pairs
template <typename E, typename I>
auto stream_kernel(int ns, int sw, int hd) {
    if constexpr (sizeof(E) == 4) {  // pick_wide: two stages
        if constexpr (sizeof(I) == 8) {
            if (wide_slot_bytes(8, hd) == 8) return decode_wide_kernel<I, 2, 0, int64_t>;
        }
        return sw == 64 ? decode_wide_kernel<I, 2, 64> : decode_wide_kernel<I, 2>;
    } else {
        return ns == 3 ? decode_stream_kernel<E, I, 3> : decode_stream_kernel<E, I, 4>;
    }
}

template <typename E, typename I>
const void* resolve_kernel(int path, bool scalar, const DecodeArgs& a) {
    const auto kernel =
        path == kStaged
            ? ((sizeof(E) == 2 && scalar)
                   ? vec1_kernel<I, true>(a.slice_cols)
                   : vec_kernel<E, I, true>(a.slice_cols))
        : path == kStream ? stream_kernel<E, I>(a.stream_stages, a.slice_cols, a.hd)
                          : decode_simt_kernel<E, I>;
    return reinterpret_cast<const void*>(kernel);
}

constexpr int kWideRowsMin = 12;  // chunk rows of the float32 streaming kernel, at least
constexpr int kWideRowsMax = 128;  // and at most

// Geometry of decode_wide_kernel: one block per (stream, slice of up to 256 columns), a column per
// thread. Each block is a chain of dependent row fetches whose time per token is set by the round
// trips its ring needs, so the rows its ring keeps in flight (two stages of ch rows) matter most; more
// blocks per SM then keep the SM's memory traffic going while one block waits at a barrier or drains
// its ring. Among slices of 256, 128 and 64 columns (at most the row), take those that run the grid
// in the fewest waves (blocks per SM bounded by registers; the ring as deep as a block's share of the
// SM's shared memory allows, at least kWideRowsMin rows per stage), and among them the narrowest
// whose ring holds at least 85 % of the deepest one's rows.
struct WideGeometry {
    int sw, ch, ns;
};

WideGeometry pick_wide(const DecodeArgs& a, int is) {
    const int sms = sm_count();
    const size_t smem_sm = smem_per_sm(), reserve = smem_reserved_per_block();
    const int most = std::min(kWideRowsMax, std::max(std::max(a.W, a.R), kWideRowsMin));
    const int full = std::min(a.hd, 256) / 4 * 4;
    WideGeometry cand[3];
    int64_t waves[3];
    int n = 0;
    for (int w0 : {256, 128, 64}) {
        const int w = std::min(w0, full);
        if (w0 < 256 && w < w0) continue;  // the narrower row is covered by the wider candidate
        const int64_t nb = a.n_streams * ((a.hd + w - 1) / w);
        const size_t meta = WideLayout(a.W, a.R, a.G, w, 0, 4, wide_slot_bytes(is, a.hd)).total;
        int64_t per_sm = std::min<int64_t>((nb + sms - 1) / sms, 65536 / (((w + 31) / 32 * 32) * kWideRegs));
        int ns = 2, ch = 0;
        for (; per_sm >= 1; --per_sm) {  // as many blocks per SM as leave each a ring of kWideRowsMin rows
            const size_t budget = smem_sm / (size_t)per_sm;
            if (budget <= meta + reserve) continue;
            const int64_t rows = (int64_t)((budget - meta - reserve) / ((size_t)w * 4));
            ns = 2;  // two tall stages: fewer chunks, each with its two barriers and its wait
            // a multiple of 16 rows where a pass takes several chunks: 48 rather than 52 rows (256
            // streams, 0.284 vs 0.291 ms), 96 rather than 100 (128 streams, 0.162 vs 0.164 ms)
            const int c = (int)std::min<int64_t>(rows / ns, most);
            ch = c < most && c >= 16 ? c / 16 * 16 : c / 4 * 4;
            if (ch >= kWideRowsMin) break;
        }
        if (per_sm < 1) continue;
        cand[n] = WideGeometry{w, ch, ns};
        waves[n++] = (nb + per_sm * sms - 1) / (per_sm * sms);
    }
    if (n == 0) return WideGeometry{full, kWideRowsMin, 2};
    int64_t fewest = waves[0];
    int deepest = 0;
    for (int i = 0; i < n; ++i) fewest = std::min(fewest, waves[i]);
    for (int i = 0; i < n; ++i)
        if (waves[i] == fewest) deepest = std::max(deepest, cand[i].ns * cand[i].ch);
    for (int i = n - 1; i >= 0; --i)  // candidates run from the widest slice to the narrowest
        if (waves[i] == fewest && 20 * cand[i].ns * cand[i].ch >= 17 * deepest) return cand[i];
    return cand[0];
}

int shrink_cols(int sw, int q) {
    const int half = (sw / 2 + q - 1) / q * q;
    return std::max(q, half);
}

}  // namespace

int launch_decode(const DecodeArgs& a, int bank_dtype, int idx_dtype, cudaStream_t stream) {
    DecodeLaunch L;
    const int rc = plan_decode(a, bank_dtype, idx_dtype, &L);
    if (rc != 0) return rc;
    return run_decode(L, stream);
}

int run_decode(const DecodeLaunch& L, cudaStream_t stream) {
    if (L.fn == nullptr) return 0;
    DecodeArgs a = L.a;
    int early = L.early_trigger;
    void* args[] = {&a, &early};
    return launch_pdl_raw(L.fn, dim3(L.grid), dim3(L.block), L.smem, stream, args);
}

int plan_decode(const DecodeArgs& a0, int bank_dtype, int idx_dtype, DecodeLaunch* L) {
    *L = DecodeLaunch{};
    DecodeArgs a = a0;
    if (a.n_streams == 0 || a.T == 0) return 0;
    const int es = bank_dtype == SDM_BF16 ? 2 : 4;
    const int is = idx_dtype == SDM_I64 ? 8 : 4;
    const auto al = [](const void* p, uintptr_t n) { return reinterpret_cast<uintptr_t>(p) % n == 0; };
    // vector path: whole 16-byte row chunks for the bulk copies, column pairs for the threads
    const bool vec = ((int64_t)a.hd * es) % 16 == 0 && al(a.bank, 16) && al(a.out, 2 * es) && al(a.v, 8);
    const int cpt = vec ? 2 : 1;
    const int q = vec ? 16 / es : 32;  // slice granularity in columns
    const int maxwr = std::max(a.W, a.R);

    // Column slice: the whole row when it fits; narrower to bound shared memory and to give the
    // grid at least two blocks per SM when there are few streams. When staging every row would
    // force slices narrower than 256 bytes (wide rows with many writes or reads), the rows stream
    // through a chunk ring instead, with slices of up to 512 bytes (or whole rows of up to 1 KiB,
    // chosen below).
    const int full = vec ? std::min(a.hd, kMaxThreads * cpt) / q * q : std::min(a.hd, kMaxThreads * cpt);
    int sw = full;
    while ((size_t)maxwr * sw * es > kRowsBudget && sw > q) sw = shrink_cols(sw, q);
    const bool streamed = vec && (int64_t)sw * es < std::min<int64_t>((int64_t)full * es, 256);
    if (streamed) sw = std::min(full, 512 / es) / q * q;
    const int64_t want_blocks = 2LL * sm_count();
    while (a.n_streams * ((a.hd + sw - 1) / sw) < want_blocks && sw * es > 128) {
        const int next = shrink_cols(sw, q);
        if (next >= sw) break;
        sw = next;
    }
    a.slice_cols = sw;
    a.n_slices = (a.hd + sw - 1) / sw;
    const int64_t blocks = a.n_streams * a.n_slices;
    if (blocks > INT_MAX) return SDM_ECOUNT;
    // decay-and-write by 16-byte pieces on every grid: one more barrier per token, a quarter of the
    // per-row stores and address work (serving workload 0.528 vs 0.541 ms, 304 streams 0.334 vs
    // 0.344, 456 streams 0.367 vs 0.379, the prompt of 64 streams 4.45 vs 4.86 ms)
    a.piece_write = 1;
    a.stream_rows = kStreamRowsMin;
    a.stream_stages = 4;
    if (streamed && es == 4) {  // float32: the slice geometry of decode_wide_kernel
        const WideGeometry g = pick_wide(a, is);
        sw = g.sw;
        a.stream_rows = g.ch;
        a.stream_stages = g.ns;
        a.slice_cols = sw;
        a.n_slices = (a.hd + sw - 1) / sw;
        if (a.n_streams * a.n_slices > INT_MAX) return SDM_ECOUNT;
    } else if (streamed) {
        // the largest chunk that keeps the whole grid resident in one wave, for slices of w columns
        // and a ring of ns chunks
        const auto chunk_rows = [&](int w, int64_t nb, int ns) {
            const int64_t per_sm = (nb + sm_count() - 1) / sm_count();
            const size_t meta = StreamLayout(a.W, a.R, a.G, w, es, is, 0, ns).total;
            const size_t block_budget = smem_per_sm() / (size_t)per_sm;
            const size_t reserve = smem_reserved_per_block();
            const size_t stage_row = (size_t)ns * w * es;
            if (block_budget <= meta + reserve) return kStreamRowsMin;
            const int64_t fit = (int64_t)((block_budget - meta - reserve) / stage_row);
            const int most = std::min(kStreamRowsMax, std::max(maxwr, kStreamRowsMin));
            return (int)std::max<int64_t>(kStreamRowsMin, std::min<int64_t>(fit, most));
        };
        // The slices as chosen above, or whole rows of up to 1 KiB instead when that keeps as many
        // SMs busy and gives a taller chunk: the rows in flight per row of work grow with the
        // chunk height (e.g. 256 streams of 1 KiB rows: 256 blocks with 32-row chunks instead of
        // 512 blocks of half rows with 25).
        const int wide = std::min(full, 1024 / es) / q * q;
        const auto geometry = [&](int ns, int& w, int& ch) {
            w = sw;
            ch = chunk_rows(sw, blocks, ns);
            if (wide > sw && a.hd <= wide) {
                const int64_t busy = std::min<int64_t>(blocks, sm_count());
                const int64_t busy_wide = std::min<int64_t>(a.n_streams, sm_count());
                const int chw = chunk_rows(wide, a.n_streams, ns);
                if (busy_wide >= busy && chw > ch) {
                    w = wide;
                    ch = chw;
                }
            }
        };
        int w = sw, ch = kStreamRowsMin;
        geometry(3, w, ch);
        if (ch >= kTallChunk) {
            a.stream_stages = 3;
        } else {
            geometry(4, w, ch);
        }
        sw = w;
        a.slice_cols = sw;
        a.n_slices = (a.hd + sw - 1) / sw;
        a.stream_rows = ch;
    }
    const int64_t blocks_final = a.n_streams * a.n_slices;
    const int path = !vec ? kSimt : streamed ? kStream : kStaged;
    // One column per thread (scalar chains, twice the warps): float32 streaming (decode_wide_kernel),
    // and bf16 staged slices of up to 64 columns, the narrow slices of grids with few streams, which
    // wait on latency and gain from the extra warps (full 256-byte rows of many streams keep
    // column pairs: 7 % faster there).
    const bool scalar = (path == kStream && es == 4) || (path == kStaged && es == 2 && sw <= 64);
    const int tcols = scalar ? 1 : cpt;
    const int threads = ((sw + tcols - 1) / tcols + 31) / 32 * 32;
    const size_t smem = path == kStaged ? VecLayout(a.W, a.R, a.G, sw, es, is).total
                        : path == kStream
                            ? (es == 4 ? WideLayout(a.W, a.R, a.G, sw, a.stream_rows, a.stream_stages, wide_slot_bytes(is, a.hd)).total
                                       : StreamLayout(a.W, a.R, a.G, sw, es, is, a.stream_rows, a.stream_stages).total)
                            : SimtLayout(a.W, a.R, sw, es).total;

    const void* fn = bank_dtype == SDM_BF16
                         ? (idx_dtype == SDM_I32 ? resolve_kernel<uint16_t, int32_t>(path, scalar, a)
                                                 : resolve_kernel<uint16_t, int64_t>(path, scalar, a))
                         : (idx_dtype == SDM_I32 ? resolve_kernel<float, int32_t>(path, scalar, a)
                                                 : resolve_kernel<float, int64_t>(path, scalar, a));
    const int rc = allow_smem(fn, smem);  // before the occupancy query
    if (rc != 0) return rc;
    // the early trigger only when every block of this launch is resident at once, so that blocks
    // of the next kernel scheduled early cannot take the place of blocks of this one
    L->early_trigger = blocks_final <= (int64_t)blocks_per_sm(fn, threads, smem) * sm_count() ? 1 : 0;
    L->fn = fn;
    L->a = a;
    L->grid = (unsigned)blocks_final;
    L->block = (unsigned)threads;
    L->smem = smem;
    return 0;
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
