// ulysses.cu - head <-> sequence relayout around the Ulysses all-to-all
// ("Ulysses relayout", TeleFuser PR #23 "Changes Made"; "Fuse Q/K RMSNorm,
// RoPE, and Ulysses packing", TeleFuser PR #38 section 2).
//
// pack:   src [rows, row_stride] holding H heads of D values per row
//         -> dst [G][rows][H/G][D]: block g is what sequence-parallel rank g
//            receives (heads g*H/G .. (g+1)*H/G - 1 of every local token).
// unpack: the inverse, [G][rows][H/G][D] -> [rows, row_stride].
//
// A bit-exact permutation, HBM-bound (2 bytes read + 2 written per element).
// One CTA walks whole token rows; the row side of every access is
// contiguous, the head side is contiguous in runs of D values.
#include "common.cuh"
#include "kernels.h"

namespace tfk {
namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) relayout_kernel(const uint16_t* __restrict__ src,
                                                            uint16_t* __restrict__ dst, int64_t row_stride,
                                                            int64_t rows, int n_heads, int head_dim,
                                                            int heads_per_group, int pack) {
    const int vec_per_head = head_dim >> 3;
    const int vec_per_row = n_heads * vec_per_head;
    const int64_t group_elems = rows * (int64_t)heads_per_group * head_dim;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        for (int v = threadIdx.x; v < vec_per_row; v += kThreads) {
            const int h = v / vec_per_head;
            const int e = v - h * vec_per_head;
            const int g = h / heads_per_group;
            const int hl = h - g * heads_per_group;
            const int64_t row_off = r * row_stride + (int64_t)v * 8;
            const int64_t grp_off = g * group_elems + (r * heads_per_group + hl) * (int64_t)head_dim + e * 8;
            if (pack)
                st_vec(dst + grp_off, ld_ro(src + row_off));
            else
                st_vec(dst + row_off, ld_ro(src + grp_off));
        }
    }
}

}  // namespace

cudaError_t launch_ulysses_relayout(const uint16_t* src, uint16_t* dst, int64_t row_stride, int64_t rows,
                                    int n_heads, int head_dim, int groups, bool pack, cudaStream_t stream) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    const void* fn = reinterpret_cast<const void*>(&relayout_kernel);
    const int per_sm = blocks_per_sm(fn, kThreads, 0);
    if (per_sm <= 0) return cudaErrorInvalidConfiguration;
    int64_t grid = (int64_t)per_sm * di.sm_count * 4;
    if (grid > rows) grid = rows;
    relayout_kernel<<<(unsigned)grid, kThreads, 0, stream>>>(src, dst, row_stride, rows, n_heads, head_dim,
                                                             n_heads / groups, pack ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace tfk
