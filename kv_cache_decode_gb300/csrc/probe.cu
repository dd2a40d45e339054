// Read-only streaming probe: the rate at which one pass over a buffer that is
// only read reaches shared memory, moved the way the attention kernels move
// the KV cache (bulk asynchronous copies into a ring of shared-memory stages,
// one CTA per SM, each CTA a contiguous slice). The result is the practical
// ceiling for a kernel that reads N bytes once: launch, first-data latency
// and drain are part of it, as they are part of every attention launch.
//
// Decode attention is bound by reading the KV cache (Efficiently Scaling
// Transformer Inference, section 2; All About Transformer Inference, "What
// about attention?"), so this read rate, beside the copy bandwidth, is the
// roofline the attention kernels are measured against.
#include <cuda_runtime.h>

#include <atomic>

#include "../../include/kvdecode.h"
#include "common.cuh"
#include "tc_common.cuh"

namespace kvd {
namespace {

constexpr int kStageBytes = 32 * 1024;
constexpr int kStages = 6;
constexpr int kSmem = kStageBytes * kStages;

// One thread per CTA issues the copies; each stage is reused once its
// previous copy has landed. Waits are bounded (~2 s of clock cycles); a
// timeout sets KVD_STATUS_TIMEOUT and the thread waits (bounded again) for
// its copies in flight before it leaves.
__global__ void __launch_bounds__(32, 1)
    read_probe_kernel(const uint8_t* __restrict__ src, unsigned long long units16,
                      unsigned long long* __restrict__ sink, int32_t* status) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kStages];
    __shared__ int abort_flag;
    constexpr long long kBudget = 4000000000LL;
    if (threadIdx.x != 0) return;
    const unsigned long long c = blockIdx.x, C = gridDim.x;
    const unsigned long long lo = units16 * c / C * 16, hi = units16 * (c + 1) / C * 16;
    const uint32_t sbase = smem_u32(smem), bbase = smem_u32(bars);
    for (int s = 0; s < kStages; ++s) tc::mbar_init(bbase + 8u * s, 1);
    abort_flag = 0;
    tc::mbar_fence_init();
    volatile int* abort_p = &abort_flag;
    const uint64_t pol = l2_evict_first_policy();
    const unsigned long long n = (hi - lo + kStageBytes - 1) / kStageBytes;
    unsigned long long acc = 0, j = 0;
    for (; j < n; ++j) {
        const int s = (int)(j % kStages);
        const uint32_t bar = bbase + 8u * s;
        if (j >= kStages) {
            if (!tc::mbar_wait(bar, (uint32_t)((j / kStages - 1) & 1), abort_p, kBudget)) break;
            acc += *reinterpret_cast<const unsigned long long*>(smem + s * kStageBytes);
        }
        const unsigned long long off = lo + j * kStageBytes;
        const uint32_t bytes = (uint32_t)((hi - off) < (unsigned long long)kStageBytes ? (hi - off) : kStageBytes);
        tc::mbar_arrive_expect_tx(bar, bytes);
        tc::bulk_load_1d(sbase + (uint32_t)(s * kStageBytes), src + off, bytes, bar, pol);
    }
    // Do not leave with copies in flight.
    for (unsigned long long jj = (j > kStages ? j - kStages : 0); jj < j; ++jj) {
        const int s = (int)(jj % kStages);
        if (tc::mbar_wait(bbase + 8u * s, (uint32_t)((jj / kStages) & 1), abort_p, kBudget / 4))
            acc += *reinterpret_cast<const unsigned long long*>(smem + s * kStageBytes);
    }
    if (*abort_p && status) atomicOr(status, KVD_STATUS_TIMEOUT);
    if (sink) sink[c] = acc;
}

constexpr int kMaxDevices = 64;
std::atomic<bool> g_probe_ready[kMaxDevices];

}  // namespace
}  // namespace kvd

extern "C" kvd_status kvd_probe_read(const void* src, size_t bytes, int ctas, unsigned long long* sink,
                                     int32_t* status_word, kvd_stream_t stream) {
    using namespace kvd;
    if (!src || ctas < 0 || (reinterpret_cast<uintptr_t>(src) & 15) || (reinterpret_cast<uintptr_t>(sink) & 7) ||
        (reinterpret_cast<uintptr_t>(status_word) & 3))
        return KVD_ERR_INVALID_ARG;
    if (bytes < 16) return KVD_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVD_ERR_CUDA;
    if (ctas == 0 && cudaDeviceGetAttribute(&ctas, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return KVD_ERR_CUDA;
    if (!g_probe_ready[dev].load(std::memory_order_acquire)) {
        if (cudaFuncSetAttribute(read_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem) !=
            cudaSuccess)
            return KVD_ERR_CUDA;
        g_probe_ready[dev].store(true, std::memory_order_release);
    }
    read_probe_kernel<<<ctas, 32, kSmem, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(src), (unsigned long long)(bytes / 16), sink, status_word);
    return cudaGetLastError() == cudaSuccess ? KVD_OK : KVD_ERR_CUDA;
}
