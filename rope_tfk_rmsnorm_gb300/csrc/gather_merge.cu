// gather_merge.cu - valid-only gather and zero-tail merge (TeleFuser PR #38,
// section 2: the gather of the valid rows fused with the merge that writes
// them back and zeroes the tail).
//
// Both buffers have contiguous rows, so the valid prefix of L rows is one
// contiguous run of L*hidden bf16 values: the gather is a bit-exact 16-byte
// vector copy, and the merge is the same copy followed, in the same launch,
// by +0.0 stores over the tail rows (no separate memset pass).
//
// Design (HBM-bound): grid-stride over 16-byte vectors, U independent loads
// per thread before the stores, full-occupancy 256-thread CTAs.
#include "common.cuh"
#include "kernels.h"

namespace tfk {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kThreads) copy_zero_kernel(const Vec8* __restrict__ src,
                                                             Vec8* __restrict__ dst, int64_t n_copy,
                                                             int64_t n_total) {
    const int64_t step = (int64_t)gridDim.x * kThreads * kUnroll;
    grid_dep_wait();
    for (int64_t base = (int64_t)blockIdx.x * kThreads * kUnroll + threadIdx.x; base < n_total;
         base += step) {
        Vec8 v[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const int64_t i = base + (int64_t)k * kThreads;
            if (i < n_copy) {
                v[k] = ld_ro(src + i);
            } else {
                v[k].w[0] = v[k].w[1] = v[k].w[2] = v[k].w[3] = 0u;  // +0.0 bf16
            }
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const int64_t i = base + (int64_t)k * kThreads;
            if (i < n_total) st_vec(dst + i, v[k]);
        }
    }
}

cudaError_t launch_copy_zero(const uint16_t* src, uint16_t* dst, int64_t n_copy, int64_t n_total,
                             cudaStream_t stream) {
    if (n_total <= 0) return cudaSuccess;
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    const void* fn = reinterpret_cast<const void*>(&copy_zero_kernel);
    const int per_sm = blocks_per_sm(fn, kThreads, 0);
    if (per_sm <= 0) return cudaErrorInvalidConfiguration;
    const int64_t per_block = (int64_t)kThreads * kUnroll;
    int64_t grid = (int64_t)per_sm * di.sm_count * 4;
    const int64_t need = (n_total + per_block - 1) / per_block;
    if (grid > need) grid = need;
    return launch_kernel(copy_zero_kernel, (unsigned)grid, kThreads, 0, stream,
                         reinterpret_cast<const Vec8*>(src), reinterpret_cast<Vec8*>(dst), n_copy, n_total);
}

}  // namespace

cudaError_t launch_valid_gather(const uint16_t* padded, uint16_t* compact, int64_t n_vec,
                                cudaStream_t stream) {
    return launch_copy_zero(padded, compact, n_vec, n_vec, stream);
}

cudaError_t launch_zero_tail_merge(const uint16_t* compact, uint16_t* padded, int64_t n_valid_vec,
                                   int64_t n_total_vec, cudaStream_t stream) {
    return launch_copy_zero(compact, padded, n_valid_vec, n_total_vec, stream);
}

}  // namespace tfk
