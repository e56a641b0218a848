// rtp_tp_mlp_noalloc: the tensor-parallel MLP for callers that cannot
// allocate device memory.
//
// Some callers of this library may not call cudaMalloc, or anything that
// allocates device memory:
//   * code that runs inside another runtime's memory pool, where all device
//     memory belongs to that pool's allocator, so a direct allocation would
//     bypass its accounting or exceed its budget;
//   * serving loops whose memory plan is fixed at start-up and must not grow
//     while requests run.
// They still own their inputs (X and the weight shards) and their output (Z),
// but they cannot provide the intermediate GELU activations Y. This entry point
// keeps Y in a file-scope static device array of fixed size instead, then runs
// the same kernels as rtp_tp_mlp with the reduction fused into the row-parallel
// GEMM (no partial buffers).
//
// The array costs kStaticScratchBytes of device memory on every GPU where this
// library's code for it is loaded, until the process exits.
#include <cuda_runtime.h>

#include <atomic>

#include "rtp_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = 16u << 20;  // 16 MiB: room for P * M * (F/P) bf16 activations
constexpr size_t kAlign = 256;

static __device__ __align__(256) unsigned char g_tp_static_scratch[kStaticScratchBytes];

// Device address of the array, per device, found once with that device current
// (threads racing on a first call find the same address). The address belongs
// to the device's context at that time: after a device reset
// (cudaDeviceReset) the module is loaded again and the array may move, so this
// entry point does not support a reset after its first call on a device.
std::atomic<void*> g_scratch_addr[64];

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

}  // namespace

extern "C" int rtp_tp_mlp_noalloc(int P, int64_t M, int64_t K, int64_t F, int64_t N, const void* X,
                                  const void* const* A_shards, const void* const* B_shards, float* Z,
                                  rtp_stream stream)
{
    const char* fn = "rtp_tp_mlp_noalloc";
    if (P < 1 || P > 8) return rtp::fail(RTP_EUNSUPPORTED, "%s: P = %d outside [1, 8]", fn, P);
    if (M < 0 || K < 1 || F < 1 || N < 1 || F % P)
        return rtp::fail(RTP_ESHAPE, "%s: sizes M=%lld K=%lld F=%lld N=%lld P=%d", fn, (long long)M, (long long)K,
                         (long long)F, (long long)N, P);
    // Checked factor by factor first, so that no product below can wrap: each
    // rank's activations must fit the array on their own before M x F/P is formed.
    const size_t Fp = (size_t)(F / P);
    if ((size_t)M > kStaticScratchBytes / 2 || Fp > kStaticScratchBytes / 2 ||
        (M > 0 && (size_t)M * Fp > kStaticScratchBytes / 2))
        return rtp::fail(RTP_ESHAPE,
                         "%s: M=%lld x F/P=%zu bf16 activations of one rank exceed the static scratch of %zu bytes",
                         fn, (long long)M, Fp, kStaticScratchBytes);
    const size_t per_rank = round_up((size_t)M * Fp * 2u);
    if (per_rank > kStaticScratchBytes / (size_t)P)
        return rtp::fail(RTP_ESHAPE,
                         "%s: the GELU activations need %zu bytes (M x F bf16, each rank padded to %zu bytes); "
                         "the static scratch holds %zu bytes (M x F <= about %zu elements)",
                         fn, per_rank * (size_t)P, kAlign, kStaticScratchBytes, kStaticScratchBytes / 2);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return rtp::fail(RTP_ECUDA, "%s: cudaGetDevice: %s", fn, cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return rtp::fail(RTP_EUNSUPPORTED, "%s: device %d", fn, dev);
    void* addr = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!addr) {
        // Set-up, once per device, with that device current. In host code the
        // array's name is only a stand-in, so the kernels get this address.
        e = cudaGetSymbolAddress(&addr, g_tp_static_scratch);
        if (e != cudaSuccess || !addr)
            return rtp::fail(RTP_ECUDA, "%s: cudaGetSymbolAddress: %s", fn, cudaGetErrorString(e));
        g_scratch_addr[dev].store(addr, std::memory_order_release);
    }
    char* base = static_cast<char*>(addr);
    void* Y[8];
    for (int i = 0; i < P; ++i) Y[i] = base + (size_t)i * per_rank;
    // The same path as rtp_tp_mlp, fused reduction, one stream. Y is written
    // in full by the first GEMM before the second reads it, so nothing in the
    // array needs clearing between calls.
    return rtp_tp_mlp(P, M, K, F, N, X, A_shards, B_shards, Y, nullptr, Z, 1, 1, 1, stream, stream);
}
