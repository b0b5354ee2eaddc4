// read_stream.cu -- a plain streaming read of device memory (a measurement aid).
//
// Decode attention is a read stream: nearly all of its bytes are KV tiles read
// once.  The copy rate usually quoted as the memory peak counts reads and
// writes together, so a pure read stream can exceed it.  This kernel reads a
// buffer once with 16-byte vector loads, eight independent loads in flight
// per thread over a grid of a few CTAs per SM, and folds the data into one
// word so the loads cannot be dropped: its rate is the practical read peak
// the attention kernels are compared with.  It also serves to evict the L2
// (reading more than the L2 holds leaves it full of clean, unrelated lines).
#include "../../include/pkv.h"
#include "pkv_internal.h"

namespace pkv {

constexpr int kReadThreads = 512;
constexpr int kReadUnroll = 8;

__global__ void __launch_bounds__(kReadThreads)
    read_stream_kernel(const uint4* __restrict__ p, size_t n16, unsigned* __restrict__ sink) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    unsigned acc = 0;
    for (; i + (kReadUnroll - 1) * stride < n16; i += kReadUnroll * stride) {
        uint4 v[kReadUnroll];
#pragma unroll
        for (int k = 0; k < kReadUnroll; ++k) v[k] = __ldg(p + i + k * stride);
#pragma unroll
        for (int k = 0; k < kReadUnroll; ++k) acc ^= v[k].x ^ v[k].y ^ v[k].z ^ v[k].w;
    }
    for (; i < n16; i += stride) {
        const uint4 v = __ldg(p + i);
        acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, off);
    if ((threadIdx.x & 31) == 0) atomicXor(sink, acc);
}

}  // namespace pkv

extern "C" int pkv_read_stream(const void* buf, size_t bytes, unsigned* sink, int ctas_per_sm,
                               void* stream) {
    if (!buf || !sink || bytes % 16 != 0 || ctas_per_sm < 1 || ctas_per_sm > 4 ||
        reinterpret_cast<uintptr_t>(buf) % 16 != 0 || reinterpret_cast<uintptr_t>(sink) % 4 != 0)
        return PKV_ERR_INVALID_ARG;
    if (bytes == 0) return PKV_OK;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
        return PKV_ERR_CUDA;
    pkv::read_stream_kernel<<<sms * ctas_per_sm, pkv::kReadThreads, 0,
                              static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(buf), bytes / 16, sink);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
