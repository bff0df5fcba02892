/*
 * Host generator of the synthetic per-step inputs (see gen_rules.h for the
 * rules).  Built into libclkgen_host.so.  The entry points fill one logit row
 * or one step's head proposals; their signatures match the input-provider
 * callbacks of the CPU oracle, which receives them as plain function
 * pointers together with a pointer to a wl_ctx.
 */
#include <stddef.h>
#include <stdint.h>

#include "gen_rules.h"

enum { WL_BF16 = 0, WL_F32 = 1 };

/* Everything a request's inputs depend on.  `stream` holds, per request, the
 * prompt followed by the ground-truth continuation (CSR by `stream_off`). */
typedef struct wl_ctx {
    uint64_t seed;
    int32_t V;
    int32_t dtype; /* WL_BF16 or WL_F32 */
    int32_t B;
    int32_t pad;
    const int32_t* stream;
    const int64_t* stream_off; /* B + 1 offsets */
    const uint16_t* t0_bf16;   /* 65,536 entries, bf16 bits */
    const uint16_t* t8_bf16;
    const float* t0_f32;
    const float* t8_f32;
} wl_ctx;

/* Ground-truth token of request b at absolute position P, or -1 past the end. */
int32_t wl_truth(const wl_ctx* c, int32_t b, int64_t P)
{
    int64_t len = c->stream_off[b + 1] - c->stream_off[b];
    if (P < 0 || P >= len) return -1;
    return c->stream[c->stream_off[b] + P];
}

/* Fill `out` with the V logits of request b at absolute position P. */
void wl_logits_row(const void* ctx, int32_t b, int64_t P, void* out)
{
    const wl_ctx* c = (const wl_ctx*)ctx;
    const uint64_t key = wl_row_key(c->seed, (uint32_t)b, (uint64_t)P);
    const int32_t truth = wl_truth(c, b, P);
    if (c->dtype == WL_BF16) {
        uint16_t* o = (uint16_t*)out;
        for (int32_t v = 0; v < c->V; ++v) {
            uint32_t idx = wl_logit_index(key, (uint32_t)v);
            o[v] = (v == truth) ? c->t8_bf16[idx] : c->t0_bf16[idx];
        }
    } else {
        float* o = (float*)out;
        for (int32_t v = 0; v < c->V; ++v) {
            uint32_t idx = wl_logit_index(key, (uint32_t)v);
            o[v] = (v == truth) ? c->t8_f32[idx] : c->t0_f32[idx];
        }
    }
}

/* Fill out[0..6] with the head proposals of request b at step t, whose
 * history has length n before the step. */
void wl_head(const void* ctx, int32_t b, int32_t t, int64_t n, int32_t* out)
{
    const wl_ctx* c = (const wl_ctx*)ctx;
    for (uint32_t i = 0; i < WL_HEAD; ++i) {
        uint64_t w = wl_head_word(c->seed, (uint32_t)b, (uint32_t)t, i);
        out[i] = wl_head_token(w, i, wl_truth(c, b, n + (int64_t)i), (uint32_t)c->V);
    }
}

/* Fill rows [0, rows) of a [rows, V] block for positions P0 .. P0+rows-1. */
void wl_logits_block(const void* ctx, int32_t b, int64_t P0, int32_t rows, void* out)
{
    const wl_ctx* c = (const wl_ctx*)ctx;
    size_t esz = (c->dtype == WL_BF16) ? 2 : 4;
    for (int32_t r = 0; r < rows; ++r)
        wl_logits_row(ctx, b, P0 + r, (char*)out + (size_t)r * (size_t)c->V * esz);
}

/* The 16 x 2 uniforms of step t of request b (row-major [16][2]). */
void wl_uniforms(const void* ctx, int32_t b, int32_t t, float* out)
{
    const wl_ctx* c = (const wl_ctx*)ctx;
    for (uint32_t r = 0; r < WL_ROWS; ++r)
        for (uint32_t k = 0; k < 2; ++k) out[2 * r + k] = wl_uniform(c->seed, (uint32_t)b, (uint32_t)t, r, k);
}

