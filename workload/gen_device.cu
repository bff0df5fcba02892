/*
 * Device generator of the synthetic per-step inputs (rules in gen_rules.h),
 * built into libclkgen_dev.so.  It stands in for the target model's logits
 * and the draft model's head proposals and is never part of the timed path.
 * Its own position array pos[B] tracks each request's history length: it
 * starts at the prompt length and advances by the emitted count each step.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include "gen_rules.h"

enum { WL_BF16 = 0, WL_F32 = 1 };

struct wl_dev_ctx {
    uint64_t seed;
    int32_t V;
    int32_t dtype;
    int32_t B;
    int32_t pad;
    const int32_t* stream;     /* device, CSR */
    const int64_t* stream_off; /* device, B + 1 */
    const uint16_t* t0_bf16;   /* device, 65,536 */
    const uint16_t* t8_bf16;
    const float* t0_f32;
    const float* t8_f32;
};

__device__ __forceinline__ int32_t wl_dev_truth(const wl_dev_ctx& c, int32_t b, int64_t P)
{
    int64_t o = c.stream_off[b];
    int64_t len = c.stream_off[b + 1] - o;
    if (P < 0 || P >= len) return -1;
    return c.stream[o + P];
}

/* One thread writes 8 consecutive elements of row (b, r). Grid: (x: row chunks, y: rows, z: B). */
__global__ void wl_logits_kernel(wl_dev_ctx c, const int64_t* __restrict__ pos, void* out,
                                 int64_t row_stride, int64_t req_stride, int32_t rows)
{
    const int32_t b = blockIdx.z;
    const int32_t r = blockIdx.y;
    const int64_t P = pos[b] + r;
    const uint64_t key = wl_row_key(c.seed, (uint32_t)b, (uint64_t)P);
    const int32_t truth = wl_dev_truth(c, b, P);
    const int64_t v0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
    if (v0 >= c.V) return;
    const int64_t base = (int64_t)b * req_stride + (int64_t)r * row_stride;
    if (c.dtype == WL_BF16) {
        uint16_t* o = (uint16_t*)out + base;
        #pragma unroll
        for (int e = 0; e < 8; ++e) {
            int64_t v = v0 + e;
            if (v < c.V) {
                uint32_t idx = wl_logit_index(key, (uint32_t)v);
                o[v] = (v == truth) ? c.t8_bf16[idx] : __ldg(&c.t0_bf16[idx]);
            }
        }
    } else {
        float* o = (float*)out + base;
        #pragma unroll
        for (int e = 0; e < 8; ++e) {
            int64_t v = v0 + e;
            if (v < c.V) {
                uint32_t idx = wl_logit_index(key, (uint32_t)v);
                o[v] = (v == truth) ? c.t8_f32[idx] : __ldg(&c.t0_f32[idx]);
            }
        }
    }
}

__global__ void wl_head_kernel(wl_dev_ctx c, const int64_t* __restrict__ pos, int32_t t, int32_t* out)
{
    int32_t b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= c.B) return;
    int64_t n = pos[b];
    for (uint32_t i = 0; i < WL_HEAD; ++i) {
        uint64_t w = wl_head_word(c.seed, (uint32_t)b, (uint32_t)t, i);
        out[(int64_t)b * WL_HEAD + i] = wl_head_token(w, i, wl_dev_truth(c, b, n + (int64_t)i), (uint32_t)c.V);
    }
}

__global__ void wl_advance_kernel(int64_t* pos, const int32_t* __restrict__ emitted, int32_t B)
{
    int32_t b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) pos[b] += emitted[b];
}

__global__ void wl_uniform_kernel(uint64_t seed, int32_t B, int32_t t, float* out)
{
    int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)B * WL_ROWS * 2) return;
    uint32_t b = (uint32_t)(i / (WL_ROWS * 2)), r = (uint32_t)((i / 2) % WL_ROWS), k = (uint32_t)(i % 2);
    out[i] = wl_uniform(seed, b, (uint32_t)t, r, k);
}

static int wl_check(cudaError_t e) { return e == cudaSuccess ? 0 : -3; }

extern "C" {

/* Logits for rows 0..rows-1 of every request, positions pos[b] .. pos[b]+rows-1.
 * out is [B, rows_alloc, V] with the given element strides. Returns 0 or -3. */
int wl_dev_logits(const wl_dev_ctx* c, const int64_t* d_pos, void* d_out, int64_t row_stride,
                  int64_t req_stride, int32_t rows, cudaStream_t s)
{
    if (c->B == 0 || rows == 0) return 0;
    dim3 block(256);
    dim3 grid((unsigned)((c->V + 8 * 256 - 1) / (8 * 256)), (unsigned)rows, (unsigned)c->B);
    wl_logits_kernel<<<grid, block, 0, s>>>(*c, d_pos, d_out, row_stride, req_stride, rows);
    return wl_check(cudaGetLastError());
}

/* Head proposals [B, 7] for step t at positions pos[b]. */
int wl_dev_head(const wl_dev_ctx* c, const int64_t* d_pos, int32_t t, int32_t* d_out, cudaStream_t s)
{
    if (c->B == 0) return 0;
    wl_head_kernel<<<(c->B + 127) / 128, 128, 0, s>>>(*c, d_pos, t, d_out);
    return wl_check(cudaGetLastError());
}

/* pos[b] += emitted[b]. */
int wl_dev_advance(int64_t* d_pos, const int32_t* d_emitted, int32_t B, cudaStream_t s)
{
    if (B == 0) return 0;
    wl_advance_kernel<<<(B + 127) / 128, 128, 0, s>>>(d_pos, d_emitted, B);
    return wl_check(cudaGetLastError());
}

/* The uniforms [B, 16, 2] of step t. */
int wl_dev_uniforms(const wl_dev_ctx* c, int32_t t, float* d_out, cudaStream_t s)
{
    if (c->B == 0) return 0;
    const int64_t n = (int64_t)c->B * WL_ROWS * 2;
    wl_uniform_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(c->seed, c->B, t, d_out);
    return wl_check(cudaGetLastError());
}

}  /* extern "C" */
