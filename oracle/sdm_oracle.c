/*
 * Plain CPU oracle of the sparse delta-memory (SDM) decode step, its multi-token form and the
 * token gather. TEST INFRASTRUCTURE ONLY: the unit tests, the smoke check and the benchmark's
 * CPU-baseline leg load this file's shared library; the CUDA library never does, and the two
 * share no code, header or constant.
 *
 * Sources (the "sparse-delta-memory 2.0.0" wheel pages):
 *   - decode.py, sdm_decode_step docstring: per stream, with d = exp(g),
 *       retrieved   = sum_w k_val[w] * d[w] * bank[k_idx[w]]
 *       delta_v     = beta * (v - retrieved)
 *       bank[k_w]   = d[w] * bank[k_w] + k_val[w] * delta_v
 *       readings    = sum_r q_val[r] * bank[q_idx[r]]        (read after the write)
 *     with k_val, v and q_val rounded to the bank dtype, beta and g kept in float32, the
 *     readings returned in the bank dtype; G == 1 gives one gate per token, G == W one per write.
 *   - decode.py, _sdm_decode_kernel: float32 arithmetic on the loaded rows; every write row is
 *     loaded before any is stored; the read rows are loaded after the stores.
 *   - cuda/gather_cuda.py, module docstring: out_o[t] = sum_n w_o[t,n] * bank[idx_o[t,n]] with
 *     float32 accumulation, stash[t,n] = bank[idx_0[t,n]] (raw rows of operand 0); a token whose
 *     position in its chunk is >= valid is padding: zero outputs and zero stash rows.
 *   - cuda/gather_cuda.py, token_gather_kernel: entries of a token are split over `groups` row
 *     groups, group g taking entries g, g+groups, ... in order with fmaf; the group partials
 *     are summed in order.
 *   - cuda/gather_cuda.py, the compact-snapshot variant (kpos): instead of the stash, operand 0's
 *     rows go to a snapshot of chunk * W0 rows per chunk; entry (t, n) of a live token with
 *     kpos[t, n] >= 0 stores bank[idx_0[t, n]] at snapshot row kpos[t, n] of chunk t / chunk
 *     (its first position in the chunk's sorted rows); kpos = -1 entries and padding tokens store
 *     nothing, and no other snapshot row is written.
 *
 * Readings of the pages where they leave a step open (each is listed in the design notes):
 *   - float32 -> bfloat16 is round-to-nearest-even (NaN stays NaN, made quiet).
 *   - d = exp(g) is the float32 value nearest to e^g: computed as (float)exp((double)g).
 *   - Sums run over ascending entry index, as one fmaf chain from +0.0f:
 *       acc = fmaf(x_w, row_w[c], acc), x_w = round(k_val)*d for the retrieve, round(q_val) for
 *       the read. (The gather's own kernel accumulates with fmaf; the decode page leaves the
 *       order to a reduction primitive.)
 *   - the decay-and-write is new = fmaf(kv, delta, row * d), the product rounded first.
 *   - delta = beta * (round(v) - retrieved): a subtraction then a product, both rounded.
 * This file is compiled with -ffp-contract=off so that no other product is fused.
 *
 * Layouts (all row-major, contiguous; S = n_streams):
 *   bank [n_slots, hd] (bf16 as raw uint16 bits, or float32), updated in place by decode;
 *   k_idx, k_val [S, W]; v [S, hd]; beta [S]; g [S, G]; q_idx, q_val [S, R]; out [S, hd] in the
 *   bank dtype. The multi-token form takes every per-token array with a leading [T] axis.
 * Index ranges are the caller's contract (as on the pages); `check` != 0 additionally verifies
 * that each stream's write slots are distinct and in range, returning ORACLE_EDUP / ORACLE_ERANGE.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EARG (-1)
#define ORACLE_EDUP (-2)
#define ORACLE_ERANGE (-3)
#define ORACLE_ENOMEM (-4)

enum { O_BF16 = 0, O_F32 = 1 };
enum { O_I32 = 0, O_I64 = 1 };

/* ---- bfloat16 bit helpers (bf16 is the high half of an IEEE float32) ---- */

float oracle_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

uint16_t oracle_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u); /* NaN */
    /* round to nearest, ties to even: add half an ulp minus one, plus the kept lsb */
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* elementwise forms of the two helpers above, for array pins */
void oracle_f32_to_bf16_array(const float* x, uint16_t* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_f32_to_bf16(x[i]);
}

void oracle_bf16_to_f32_array(const uint16_t* x, float* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_bf16_to_f32(x[i]);
}

/* value rounded to the bank dtype and widened back to float32 */
static float round_to_bank(float x, int bank_dtype) {
    return bank_dtype == O_BF16 ? oracle_bf16_to_f32(oracle_f32_to_bf16(x)) : x;
}

static float bank_load(const void* bank, int bank_dtype, int64_t i) {
    return bank_dtype == O_BF16 ? oracle_bf16_to_f32(((const uint16_t*)bank)[i])
                                : ((const float*)bank)[i];
}

static void bank_store(void* bank, int bank_dtype, int64_t i, float x) {
    if (bank_dtype == O_BF16)
        ((uint16_t*)bank)[i] = oracle_f32_to_bf16(x);
    else
        ((float*)bank)[i] = x;
}

static int64_t load_index(const void* p, int idx_dtype, int64_t i) {
    return idx_dtype == O_I64 ? ((const int64_t*)p)[i] : (int64_t)((const int32_t*)p)[i];
}

/* ---- decode: one token for every stream ---- */

/* Advance stream s by one token. The per-token arrays point at this token's [S, .] slab. */
static int decode_one(void* bank, int bank_dtype, int64_t n_slots, int64_t hd, const void* k_idx,
                      const float* k_val, const float* v, const float* beta, const float* g,
                      const void* q_idx, const float* q_val, void* out, int64_t s, int W, int R,
                      int G, int idx_dtype, int check, int64_t* slot, float* kv, float* d,
                      float* rows, float* delta) {
    /* step 1: write slots, rounded write weights, gates d = exp(g) in float32 */
    for (int w = 0; w < W; ++w) {
        slot[w] = load_index(k_idx, idx_dtype, s * W + w);
        kv[w] = round_to_bank(k_val[s * W + w], bank_dtype);
        d[w] = (float)exp((double)g[s * G + (G == 1 ? 0 : w)]);
        if (check) {
            if (slot[w] < 0 || slot[w] >= n_slots) return ORACLE_ERANGE;
            for (int u = 0; u < w; ++u)
                if (slot[u] == slot[w]) return ORACLE_EDUP;
        }
    }
    /* step 2: every write row, read before any write */
    for (int w = 0; w < W; ++w)
        for (int64_t c = 0; c < hd; ++c) rows[(int64_t)w * hd + c] = bank_load(bank, bank_dtype, slot[w] * hd + c);
    /* steps 3-4: retrieved = sum_w (kv_w d_w) row_w ; delta = beta (round(v) - retrieved) */
    for (int64_t c = 0; c < hd; ++c) {
        float acc = 0.0f;
        for (int w = 0; w < W; ++w) {
            float a = kv[w] * d[w];
            acc = fmaf(a, rows[(int64_t)w * hd + c], acc);
        }
        float vr = round_to_bank(v[s * hd + c], bank_dtype);
        delta[c] = beta[s] * (vr - acc);
    }
    /* step 5: decay and write, new = d_w row_w + kv_w delta, rounded to the bank dtype */
    for (int w = 0; w < W; ++w)
        for (int64_t c = 0; c < hd; ++c) {
            float decayed = rows[(int64_t)w * hd + c] * d[w];
            bank_store(bank, bank_dtype, slot[w] * hd + c, fmaf(kv[w], delta[c], decayed));
        }
    /* steps 6-7: the read, after the write; readings rounded to the bank dtype */
    for (int64_t c = 0; c < hd; ++c) {
        float acc = 0.0f;
        for (int r = 0; r < R; ++r) {
            int64_t qs = load_index(q_idx, idx_dtype, s * R + r);
            if (check && (qs < 0 || qs >= n_slots)) return ORACLE_ERANGE;
            float qv = round_to_bank(q_val[s * R + r], bank_dtype);
            acc = fmaf(qv, bank_load(bank, bank_dtype, qs * hd + c), acc);
        }
        bank_store(out, bank_dtype, s * hd + c, acc);
    }
    return ORACLE_OK;
}

/* T tokens per stream, time-major: token t's arrays start at t * S * (per-stream length).
 * Token t of every stream is applied before token t+1 of any stream; since streams own
 * private slots, this equals running each stream's T tokens on its own. T == 1 is the
 * single-token step. */
int oracle_sdm_decode_seq(void* bank, int bank_dtype, int64_t n_slots, int64_t hd, const void* k_idx,
                          const float* k_val, const float* v, const float* beta, const float* g,
                          const void* q_idx, const float* q_val, void* out, int64_t n_streams, int W,
                          int R, int G, int idx_dtype, int64_t T, int check) {
    if (!bank || !k_idx || !k_val || !v || !beta || !g || !q_idx || !q_val || !out) return ORACLE_EARG;
    if (bank_dtype != O_BF16 && bank_dtype != O_F32) return ORACLE_EARG;
    if (idx_dtype != O_I32 && idx_dtype != O_I64) return ORACLE_EARG;
    if (hd < 1 || n_slots < 1 || n_streams < 0 || T < 0) return ORACLE_EARG;
    if (W < 1 || W > 256 || R < 1 || R > 256 || (G != 1 && G != W)) return ORACLE_EARG;
    int64_t* slot = (int64_t*)malloc(sizeof(int64_t) * (size_t)W);
    float* kv = (float*)malloc(sizeof(float) * (size_t)W);
    float* d = (float*)malloc(sizeof(float) * (size_t)W);
    float* rows = (float*)malloc(sizeof(float) * (size_t)W * (size_t)hd);
    float* delta = (float*)malloc(sizeof(float) * (size_t)hd);
    int rc = ORACLE_OK;
    if (!slot || !kv || !d || !rows || !delta) rc = ORACLE_ENOMEM;
    const size_t ies = idx_dtype == O_I64 ? 8 : 4, bes = bank_dtype == O_BF16 ? 2 : 4;
    for (int64_t t = 0; t < T && rc == ORACLE_OK; ++t) {
        const char* kit = (const char*)k_idx + (size_t)(t * n_streams * W) * ies;
        const char* qit = (const char*)q_idx + (size_t)(t * n_streams * R) * ies;
        char* ot = (char*)out + (size_t)(t * n_streams * hd) * bes;
        for (int64_t s = 0; s < n_streams && rc == ORACLE_OK; ++s)
            rc = decode_one(bank, bank_dtype, n_slots, hd, kit, k_val + t * n_streams * W, v + t * n_streams * hd,
                            beta + t * n_streams, g + t * n_streams * G, qit, q_val + t * n_streams * R, ot, s,
                            W, R, G, idx_dtype, check, slot, kv, d, rows, delta);
    }
    free(slot);
    free(kv);
    free(d);
    free(rows);
    free(delta);
    return rc;
}

int oracle_sdm_decode_step(void* bank, int bank_dtype, int64_t n_slots, int64_t hd, const void* k_idx,
                           const float* k_val, const float* v, const float* beta, const float* g,
                           const void* q_idx, const float* q_val, void* out, int64_t n_streams, int W,
                           int R, int G, int idx_dtype, int check) {
    return oracle_sdm_decode_seq(bank, bank_dtype, n_slots, hd, k_idx, k_val, v, beta, g, q_idx, q_val, out,
                                 n_streams, W, R, G, idx_dtype, 1, check);
}

/* ---- token gather ---- */

static float load_weight(const void* w, int w_dtype, int64_t i) {
    return w_dtype == O_BF16 ? oracle_bf16_to_f32(((const uint16_t*)w)[i]) : ((const float*)w)[i];
}

/* out_o[t, :] for one operand of one live token, in the order fixed by `groups`. */
static void gather_token_operand(const void* bank, int bank_dtype, int64_t hd, const void* idx,
                                 const void* w, int w_dtype, int idx_dtype, int width, int64_t t,
                                 int groups, float* out_row, float* part) {
    for (int64_t c = 0; c < hd; ++c) {
        for (int gi = 0; gi < groups; ++gi) {
            float acc = 0.0f;
            for (int n = gi; n < width; n += groups) {
                int64_t slot = load_index(idx, idx_dtype, t * width + n);
                float wt = load_weight(w, w_dtype, t * width + n);
                acc = fmaf(wt, bank_load(bank, bank_dtype, slot * hd + c), acc);
            }
            part[gi] = acc;
        }
        if (groups == 1) {
            out_row[c] = part[0];
        } else {
            float sum = 0.0f;
            for (int gi = 0; gi < groups; ++gi) sum += part[gi];
            out_row[c] = sum;
        }
    }
}

/* n_ops in {1, 2}; operand 1's arguments are ignored when n_ops == 1. stash may be NULL.
 * chunk_valid, when not NULL, holds one valid count per chunk and replaces `valid`.
 * groups >= 1 selects the summation order (1: one ascending fmaf chain per column). */
int oracle_sdm_gather(const void* bank, int bank_dtype, int64_t n_slots, int64_t hd, int n_ops,
                      const void* idx0, const void* w0, float* out0, int width0, const void* idx1,
                      const void* w1, float* out1, int width1, int idx_dtype, int w_dtype, void* stash,
                      int64_t tokens, int chunk, int valid, const int32_t* chunk_valid, int groups,
                      int check) {
    if (!bank || !idx0 || !w0 || !out0) return ORACLE_EARG;
    if (n_ops != 1 && n_ops != 2) return ORACLE_EARG;
    if (n_ops == 2 && (!idx1 || !w1 || !out1)) return ORACLE_EARG;
    if (bank_dtype != O_BF16 && bank_dtype != O_F32) return ORACLE_EARG;
    if (w_dtype != O_BF16 && w_dtype != O_F32) return ORACLE_EARG;
    if (idx_dtype != O_I32 && idx_dtype != O_I64) return ORACLE_EARG;
    if (hd < 1 || n_slots < 1 || tokens < 0 || chunk < 1 || tokens % chunk != 0) return ORACLE_EARG;
    if (!chunk_valid && (valid < 0 || valid > chunk)) return ORACLE_EARG;
    if (width0 < 1 || width0 > 256 || (n_ops == 2 && (width1 < 1 || width1 > 256))) return ORACLE_EARG;
    if (groups < 1) return ORACLE_EARG;
    float* part = (float*)malloc(sizeof(float) * (size_t)groups);
    if (!part) return ORACLE_ENOMEM;
    const size_t bes = bank_dtype == O_BF16 ? 2 : 4;
    int rc = ORACLE_OK;
    for (int64_t t = 0; t < tokens && rc == ORACLE_OK; ++t) {
        int v_t = chunk_valid ? chunk_valid[t / chunk] : valid;
        if (chunk_valid && (v_t < 0 || v_t > chunk)) {
            rc = ORACLE_EARG;
            break;
        }
        int live = (int)(t % chunk) < v_t;
        for (int o = 0; o < n_ops; ++o) {
            const void* idx = o == 0 ? idx0 : idx1;
            const void* w = o == 0 ? w0 : w1;
            float* out = o == 0 ? out0 : out1;
            int width = o == 0 ? width0 : width1;
            if (!live) {
                for (int64_t c = 0; c < hd; ++c) out[t * hd + c] = 0.0f;
                continue;
            }
            if (check)
                for (int n = 0; n < width; ++n) {
                    int64_t slot = load_index(idx, idx_dtype, t * width + n);
                    if (slot < 0 || slot >= n_slots) rc = ORACLE_ERANGE;
                }
            if (rc != ORACLE_OK) break;
            gather_token_operand(bank, bank_dtype, hd, idx, w, w_dtype, idx_dtype, width, t, groups, out + t * hd,
                                 part);
        }
        if (stash && rc == ORACLE_OK) {
            for (int n = 0; n < width0; ++n) {
                char* dst = (char*)stash + (size_t)((t * width0 + n) * hd) * bes;
                if (live) {
                    int64_t slot = load_index(idx0, idx_dtype, t * width0 + n);
                    memcpy(dst, (const char*)bank + (size_t)(slot * hd) * bes, (size_t)hd * bes);
                } else {
                    memset(dst, 0, (size_t)hd * bes);
                }
            }
        }
    }
    free(part);
    return rc;
}

/* Compact snapshot (the gather's kpos form): compact is [tokens / chunk, chunk * width0, hd] in the
 * bank dtype, kpos [tokens, width0] int32. Writes only the rows kpos names for live tokens. */
int oracle_sdm_gather_kpos(const void* bank, int bank_dtype, int64_t n_slots, int64_t hd, const void* idx0,
                           int width0, int idx_dtype, const int32_t* kpos, void* compact, int64_t tokens, int chunk,
                           int valid, const int32_t* chunk_valid, int check) {
    if (!bank || !idx0 || !kpos || !compact) return ORACLE_EARG;
    if (bank_dtype != O_BF16 && bank_dtype != O_F32) return ORACLE_EARG;
    if (idx_dtype != O_I32 && idx_dtype != O_I64) return ORACLE_EARG;
    if (hd < 1 || n_slots < 1 || tokens < 0 || chunk < 1 || tokens % chunk != 0) return ORACLE_EARG;
    if (!chunk_valid && (valid < 0 || valid > chunk)) return ORACLE_EARG;
    if (width0 < 1 || width0 > 256) return ORACLE_EARG;
    const size_t bes = bank_dtype == O_BF16 ? 2 : 4;
    const int64_t crow = (int64_t)chunk * width0; /* snapshot rows per chunk */
    for (int64_t t = 0; t < tokens; ++t) {
        int v_t = chunk_valid ? chunk_valid[t / chunk] : valid;
        if (v_t < 0 || v_t > chunk) return ORACLE_EARG;
        if ((int)(t % chunk) >= v_t) continue; /* padding: stores nothing */
        for (int n = 0; n < width0; ++n) {
            int32_t kp = kpos[t * width0 + n];
            if (kp < 0) continue;
            if (kp >= crow) {
                if (check) return ORACLE_ERANGE;
                continue;
            }
            int64_t slot = load_index(idx0, idx_dtype, t * width0 + n);
            if (check && (slot < 0 || slot >= n_slots)) return ORACLE_ERANGE;
            char* dst = (char*)compact + (size_t)(((t / chunk) * crow + kp) * hd) * bes;
            memcpy(dst, (const char*)bank + (size_t)(slot * hd) * bes, (size_t)hd * bes);
        }
    }
    return ORACLE_OK;
}
