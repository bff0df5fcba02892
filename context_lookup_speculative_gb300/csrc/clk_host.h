// Host-side helpers shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "clk.h"
#include "clk_device.cuh"

struct clk_lookup {
    clk::LookupDev dev;
    void* ws;
    size_t bytes;
    int device;
    // The fused greedy verify alternates between two scratch halves (vparity)
    // so that it may start streaming while the previous one finishes; the
    // proposal lets its dependent start at once only after such a verify
    // (last_fused = kFusedGreedy), whose scratch use it then cannot disturb.
    int vparity;
    int last_fused;
};

namespace clk {

constexpr size_t kAlign = 256;
constexpr int kFusedNone = 0, kFusedGreedy = 1, kFusedSampled = 2;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Non-null and 4-byte aligned.
inline bool ok_i32(const void* p) { return p != nullptr && aligned(p, 4); }

inline int launch_status()
{
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? CLK_OK : CLK_ECUDA;
}

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? CLK_OK : CLK_ECUDA; }

inline bool handle_ok(const clk_lookup* h) { return h != nullptr && h->ws != nullptr; }

inline int check_batch(const clk_lookup* h, int32_t B)
{
    if (!handle_ok(h)) return CLK_ESTATE;
    if (B < 0 || B > h->dev.max_slots) return CLK_EINVAL;
    return CLK_OK;
}

inline int num_sms()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

}  // namespace clk
