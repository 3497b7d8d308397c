// swiglu.cu - SwiGLU on the FFN up-projection output ("SwiGLU", TeleFuser
// PR #23 "Changes Made"):  out[t,j] = bf16( silu(g) * u ),
// silu(g) = g / (1 + exp(-g)),  g = gate_up[t,j],  u = gate_up[t,ffn+j].
//
// Design (HBM-bound: 4 bytes read + 2 written per output element): every CTA
// takes one chunk of one row; each thread issues U independent 16-byte loads
// of gate and U of up before doing any arithmetic, so 32*U bytes per thread
// are in flight; full-occupancy 256-thread CTAs keep ~256 KB in flight per SM.
// exp is the fast exp2-based intrinsic; its error (a few fp32 ulp) is far
// below the bf16 rounding of the result.
#include "common.cuh"
#include "kernels.h"

namespace tfk {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kThreads) swiglu_kernel(const uint16_t* __restrict__ gate_up,
                                                          int64_t in_stride, uint16_t* __restrict__ out,
                                                          int64_t out_stride, int ffn,
                                                          int chunks_per_row, int64_t n_blocks) {
    const int nvec = ffn >> 3;
    grid_dep_wait();
    for (int64_t b = blockIdx.x; b < n_blocks; b += gridDim.x) {
        const int64_t r = b / chunks_per_row;
        const int chunk = (int)(b - r * chunks_per_row);
        const int v0 = chunk * (kThreads * kUnroll) + threadIdx.x;
        const uint16_t* g = gate_up + r * in_stride;
        const uint16_t* u = g + ffn;
        uint16_t* o = out + r * out_stride;
        Vec8 gv[kUnroll], uv[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const int v = v0 + k * kThreads;
            if (v < nvec) {
                gv[k] = ld_ro(g + v * 8);
                uv[k] = ld_ro(u + v * 8);
            }
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const int v = v0 + k * kThreads;
            if (v < nvec) {
                float gf[8], uf[8], of[8];
                unpack8(gv[k], gf);
                unpack8(uv[k], uf);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float silu = __fdividef(gf[e], 1.0f + __expf(-gf[e]));
                    of[e] = silu * uf[e];
                }
                st_vec(o + v * 8, pack8(of));
            }
        }
    }
}

}  // namespace

cudaError_t launch_swiglu(const uint16_t* gate_up, int64_t in_stride, uint16_t* out,
                          int64_t out_stride, int64_t rows, int ffn, cudaStream_t stream) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    const int nvec = ffn / 8;
    const int chunks = (nvec + kThreads * kUnroll - 1) / (kThreads * kUnroll);
    const int64_t n_blocks = rows * chunks;
    const void* fn = reinterpret_cast<const void*>(&swiglu_kernel);
    const int per_sm = blocks_per_sm(fn, kThreads, 0);
    if (per_sm <= 0) return cudaErrorInvalidConfiguration;
    // enough CTAs for several full waves; the loop covers the rest
    int64_t grid = (int64_t)per_sm * di.sm_count * 64;
    if (grid > n_blocks) grid = n_blocks;
    return launch_kernel(swiglu_kernel, (unsigned)grid, kThreads, 0, stream, gate_up, in_stride, out,
                         out_stride, ffn, chunks, n_blocks);
}

}  // namespace tfk
