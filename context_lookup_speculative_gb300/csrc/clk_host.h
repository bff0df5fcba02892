// Host-side helpers shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "clk.h"
#include "clk_device.cuh"

struct clk_lookup {
    clk::LookupDev dev;
    void* ws;
    size_t bytes;
    int device;
    // The fused greedy verify alternates between two scratch halves (vparity),
    // and so does the fused sampled verify given a caller scratch of two
    // halves (sparity), so that each may start streaming while the previous
    // one finishes; the proposal lets its dependent start at once only after
    // such a verify (last_fused = kFusedGreedy or kFusedSampledPaired), whose
    // scratch use it then cannot disturb.
    int vparity;
    int sparity;
    int last_fused;
    // Proposal launches number themselves with ptag and leave ins records
    // (what they leave complete in the index, and insertions left to the
    // next one); defer_tag is the tag of the last proposal launch (0 once a
    // call rebuilt histories or tables).  The next proposal reads those
    // records after its wait, or before it when a fused greedy verify came
    // after the recording launch (vsince = 1), which completes only after it.
    int32_t ptag;
    int32_t defer_tag;
    int vsince;
    // 1: fused verify calls are launched with nothing to overlap
    // (clk_lookup_set_alone), so no CTA of theirs starts late.
    int alone;
};

namespace clk {

constexpr size_t kAlign = 256;
constexpr int kFusedNone = 0, kFusedGreedy = 1, kFusedSampled = 2, kFusedSampledPaired = 3;

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

// Registers one CTA of the fused proposal launch (clk_propose_fuse_sched)
// takes for nlev match lengths (allocation granularity included), or -1 on
// a CUDA error.  Defined with the kernel in clk_lookup.cu.
int proposal_cta_regs(int nlev);

// Registers a CTA of `threads` threads takes when a thread uses `regs`
// registers: warps are allocated registers in units of 256 (8 a thread).
inline int cta_regs(int regs, int threads)
{
    return ((threads + 31) / 32) * (((regs + 7) / 8) * 8 * 32);
}

// CTAs of a launch of `kernel` (`threads` threads, `occ` resident per SM)
// that one fused proposal CTA keeps off its SM while both are resident: the
// SM's registers left beside the proposal CTA hold fewer of them.
inline int displaced_by_proposal_uncached(const void* kernel, int threads, int nlev, int occ)
{
    const int p = proposal_cta_regs(nlev);
    cudaFuncAttributes fa;
    int dev = 0, regs_sm = 0;
    if (p < 0 || cudaFuncGetAttributes(&fa, kernel) != cudaSuccess || cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess)
        return 0;
    const int v = cta_regs(fa.numRegs, threads);
    const int fit = v > 0 ? (regs_sm - p) / v : occ;
    return occ - (fit < 0 ? 0 : (fit > occ ? occ : fit));
}

// The same, cached per kernel (template argument), device and number of
// match lengths (calls from any host thread).
template <auto Kern>
int displaced_by_proposal(int threads, int nlev, int occ)
{
    static std::atomic<int> cache[64][CLK_MAX_K + 1];  // value + 1; 0: not yet known
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const bool cacheable = dev >= 0 && dev < 64 && nlev >= 0 && nlev <= CLK_MAX_K;
    if (cacheable) {
        const int c = cache[dev][nlev].load(std::memory_order_relaxed);
        if (c > 0) return c - 1;
    }
    const auto kern = Kern;
    const int d = displaced_by_proposal_uncached((const void*)kern, threads, nlev, occ);
    if (cacheable) cache[dev][nlev].store(d + 1, std::memory_order_relaxed);
    return d;
}

inline int num_sms()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return sms;
}

}  // namespace clk
