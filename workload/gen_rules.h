/*
 * Seeded synthetic inputs for the context-lookup speculative decoding step:
 * the per-element rules that both the host generator (gen_host.c) and the
 * device generator (gen_device.cu) evaluate, so that the two produce the same
 * bits.  Nothing here is part of the method: these are the stand-ins for the
 * target model's logits and for the draft model's 7 head proposals.
 *
 * Counter-based hashing uses the SplitMix64 output function (Steele, Lea and
 * Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014): a
 * 64-bit input is mixed by two xor-shift-multiply rounds and a final
 * xor-shift.  Every draw is a pure function of (seed, request, position or
 * step, index), so any row can be regenerated on its own.
 *
 * Logit rule.  For request b and absolute position P (row r of a verify
 * block whose first slot sits at history length n has P = n + r), element v
 * is  T0[idx]  or, when v is the ground-truth token of position P,  T8[idx],
 * with idx the top 16 bits of  mix64(row_key(b, P) + v * golden).  T0 holds
 * the 65,536 quantiles of N(0,1) at (i + 1/2) / 65536 and T8 the same plus 8,
 * rounded to the stored type.  The tables are built on the host once.
 *
 * Head rule.  At step t, for a request whose history has length n, head slot
 * i (0-based, 0..6) proposes the ground-truth token of position n + i when
 * the high 32 bits of the slot's hash word fall below
 * floor((0.90 - 0.03 i) * 2^32); otherwise it proposes the uniform token
 * floor(lo32 * V / 2^32) from the low 32 bits of the same word.
 */
#ifndef WL_GEN_RULES_H
#define WL_GEN_RULES_H

#include <stdint.h>

#if defined(__CUDACC__)
#define WL_FN __host__ __device__ static inline
#else
#define WL_FN static inline
#endif

/* Domain-separation words, one per kind of draw. */
#define WL_DOMAIN_LOGITS 0x6C6F676974730000ull
#define WL_DOMAIN_HEAD 0x6865616400000000ull
#define WL_DOMAIN_UNIFORM 0x756E69666F726D00ull
#define WL_GOLDEN 0x9E3779B97F4A7C15ull

/* Number of head proposals per step and the verify block width. */
#define WL_HEAD 7
#define WL_ROWS 16

WL_FN uint64_t wl_mix64(uint64_t x)
{
    x ^= x >> 30;
    x *= 0xBF58476D1CE4E5B9ull;
    x ^= x >> 27;
    x *= 0x94D049BB133111EBull;
    x ^= x >> 31;
    return x;
}

/* Key of one logit row: request b, absolute position P. */
WL_FN uint64_t wl_row_key(uint64_t seed, uint32_t b, uint64_t P)
{
    return wl_mix64(wl_mix64(wl_mix64(seed ^ WL_DOMAIN_LOGITS) + b) + P);
}

/* Quantile-table index of element v of the row with key `row_key`. */
WL_FN uint32_t wl_logit_index(uint64_t row_key, uint32_t v)
{
    return (uint32_t)(wl_mix64(row_key + (uint64_t)v * WL_GOLDEN) >> 48);
}

/* Hash word of head slot i at step t of request b. */
WL_FN uint64_t wl_head_word(uint64_t seed, uint32_t b, uint32_t t, uint32_t i)
{
    return wl_mix64(wl_mix64(wl_mix64(wl_mix64(seed ^ WL_DOMAIN_HEAD) + b) + t) + i);
}

/* floor((0.90 - 0.03 i) * 2^32), computed exactly in integers. */
WL_FN uint32_t wl_head_threshold(uint32_t i)
{
    int64_t pct = 90 - 3 * (int64_t)i;
    if (pct <= 0) return 0u;
    return (uint32_t)(((uint64_t)pct << 32) / 100u);
}

/* Proposal of head slot i given its hash word and the ground truth there. */
WL_FN int32_t wl_head_token(uint64_t w, uint32_t i, int32_t truth, uint32_t V)
{
    if ((uint32_t)(w >> 32) < wl_head_threshold(i) && truth >= 0) return truth;
    return (int32_t)(((w & 0xFFFFFFFFull) * (uint64_t)V) >> 32);
}

/* Uniform number k (0: acceptance, 1: draw) of verify row r at step t of
 * request b, for sampling verification: the top 24 bits of a hash word times
 * 2^-24, a float in [0, 1) that both sides compute exactly. */
WL_FN float wl_uniform(uint64_t seed, uint32_t b, uint32_t t, uint32_t r, uint32_t k)
{
    const uint64_t w =
        wl_mix64(wl_mix64(wl_mix64(wl_mix64(seed ^ WL_DOMAIN_UNIFORM) + b) + t) + (uint64_t)(2u * r + k));
    return (float)(uint32_t)(w >> 40) * (1.0f / 16777216.0f);
}

#endif /* WL_GEN_RULES_H */
