// swiglu.cu - SwiGLU on the FFN up-projection output (TeleFuser PR #23,
// section Changes Made, its SwiGLU kernel):  out[t,j] = bf16( silu(g) * u ),
// silu(g) = g / (1 + exp(-g)),  g = gate_up[t,j],  u = gate_up[t,ffn+j].
//
// Design (HBM-bound: 4 bytes read + 2 written per output element): every CTA
// takes one chunk of one row, or several whole rows when a row is shorter
// than half a chunk (ffn <= 4096); each thread issues U independent 16-byte loads
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

// silu(g) * u for one 16-byte vector of each, stored at o.
__device__ __forceinline__ void swiglu_vec(uint16_t* o, const Vec8& gv, const Vec8& uv) {
    float gf[8], uf[8], of[8];
    unpack8(gv, gf);
    unpack8(uv, uf);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float silu = __fdividef(gf[e], 1.0f + __expf(-gf[e]));
        of[e] = silu * uf[e];
    }
    st_vec(o, pack8(of));
}

// rows_per_block == 1: block b covers chunk (b % chunks_per_row) of row
// b / chunks_per_row.  rows_per_block > 1 (rows shorter than half a chunk):
// block b covers rows [b * rows_per_block, ...), its kThreads * kUnroll
// vector slots laid over those rows back to back; a thread's (row, vector)
// positions are the same in every block and computed once.
template <bool kMultiRow>
__global__ void __launch_bounds__(kThreads) swiglu_kernel(const uint16_t* __restrict__ gate_up,
                                                          int64_t in_stride, uint16_t* __restrict__ out,
                                                          int64_t out_stride, int64_t rows, int ffn,
                                                          int chunks_per_row, int rows_per_block,
                                                          int64_t n_blocks) {
    const int nvec = ffn >> 3;
    grid_dep_wait();
    if constexpr (kMultiRow) {
        int roff[kUnroll], vv[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const int lin = threadIdx.x + k * kThreads;
            roff[k] = lin / nvec;
            vv[k] = lin - roff[k] * nvec;
            if (roff[k] >= rows_per_block) roff[k] = -1;
        }
        for (int64_t b = blockIdx.x; b < n_blocks; b += gridDim.x) {
            const int64_t row0 = b * rows_per_block;
            Vec8 gv[kUnroll], uv[kUnroll];
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int64_t r = row0 + roff[k];
                if (roff[k] >= 0 && r < rows) {
                    const uint16_t* g = gate_up + r * in_stride + vv[k] * 8;
                    gv[k] = ld_ro(g);
                    uv[k] = ld_ro(g + ffn);
                }
            }
#pragma unroll
            for (int k = 0; k < kUnroll; ++k) {
                const int64_t r = row0 + roff[k];
                if (roff[k] >= 0 && r < rows) swiglu_vec(out + r * out_stride + vv[k] * 8, gv[k], uv[k]);
            }
        }
    } else {
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
            if (v < nvec) swiglu_vec(o + v * 8, gv[k], uv[k]);
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
    // rows shorter than half a chunk: several whole rows per block
    const int rows_per_block = 2 * nvec <= kThreads * kUnroll ? (kThreads * kUnroll) / nvec : 1;
    const int64_t n_blocks = rows_per_block > 1 ? (rows + rows_per_block - 1) / rows_per_block : rows * chunks;
    const void* fn = rows_per_block > 1 ? reinterpret_cast<const void*>(&swiglu_kernel<true>)
                                        : reinterpret_cast<const void*>(&swiglu_kernel<false>);
    const int per_sm = blocks_per_sm(fn, kThreads, 0);
    if (per_sm <= 0) return cudaErrorInvalidConfiguration;
    // enough CTAs for several full waves; the loop covers the rest
    int64_t grid = (int64_t)per_sm * di.sm_count * 64;
    if (grid > n_blocks) grid = n_blocks;
    return launch_kernel(rows_per_block > 1 ? swiglu_kernel<true> : swiglu_kernel<false>, (unsigned)grid,
                         kThreads, 0, stream, gate_up, in_stride, out, out_stride, rows, ffn, chunks,
                         rows_per_block, n_blocks);
}

}  // namespace tfk
