// ulysses.cu - head <-> sequence relayout around the Ulysses all-to-all
// (TeleFuser PR #23, section Changes Made: the Ulysses relayout kernel;
// TeleFuser PR #38, section 2: the packing fused into Q/K norm and RoPE).
//
// pack:   src [rows, row_stride] holding H heads of D values per row
//         -> dst [G][rows][H/G][D]: block g is what sequence-parallel rank g
//            receives (heads g*H/G .. (g+1)*H/G - 1 of every local token).
// unpack: the inverse, [G][rows][H/G][D] -> [rows, row_stride].
//
// A bit-exact permutation, HBM-bound (2 bytes read + 2 written per element).
// CTAs over 4-row tiles; at every row the row side of a warp's accesses is
// contiguous and the grouped side contiguous in runs of (heads per group) * D
// values.
#include "common.cuh"
#include "kernels.h"

namespace tfk {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerStep = 4;
constexpr int64_t kRowsPerCta = 4;

// Each thread owns fixed 16-byte column vectors of the row layout (their
// head / group coordinates are computed once) and walks this CTA's run of
// rows, kRowsPerStep rows at a time with independent loads in flight.
__global__ void __launch_bounds__(kThreads) relayout_kernel(const uint16_t* __restrict__ src,
                                                            uint16_t* __restrict__ dst, int64_t row_stride,
                                                            int64_t rows, int n_heads, int head_dim,
                                                            int heads_per_group, int pack) {
    const int vec_per_head = head_dim >> 3;
    const int vec_per_row = n_heads * vec_per_head;
    const int64_t grp_row = (int64_t)heads_per_group * head_dim;  // elements per row inside a group
    const int64_t group_elems = rows * grp_row;
    const int64_t r0 = rows * (int64_t)blockIdx.x / gridDim.x;
    const int64_t r1 = rows * (int64_t)(blockIdx.x + 1) / gridDim.x;
    grid_dep_wait();
    for (int v = threadIdx.x; v < vec_per_row; v += kThreads) {
        const int h = v / vec_per_head;
        const int e = v - h * vec_per_head;
        const int g = h / heads_per_group;
        const int hl = h - g * heads_per_group;
        const int64_t row_col = (int64_t)v * 8;                                   // row layout
        const int64_t grp_col = g * group_elems + (int64_t)hl * head_dim + e * 8;  // grouped layout
        const int64_t row_step = pack ? row_stride : grp_row;
        const int64_t dst_step = pack ? grp_row : row_stride;
        const uint16_t* s0 = src + (pack ? row_col : grp_col);
        uint16_t* d0 = dst + (pack ? grp_col : row_col);
        int64_t r = r0;
        for (; r + kRowsPerStep <= r1; r += kRowsPerStep) {
            Vec8 t[kRowsPerStep];
#pragma unroll
            for (int k = 0; k < kRowsPerStep; ++k) t[k] = ld_ro(s0 + (r + k) * row_step);
#pragma unroll
            for (int k = 0; k < kRowsPerStep; ++k) st_vec(d0 + (r + k) * dst_step, t[k]);
        }
        for (; r < r1; ++r) st_vec(d0 + r * dst_step, ld_ro(s0 + r * row_step));
    }
}

// Rows outer, columns inner: a thread owns NV column vectors of the row layout
// (NV = ceil(vectors per row / kThreads) <= 4, coordinates computed once) and
// moves kRowsPerStep whole rows per step, so a CTA reads (pack) or writes
// (unpack) complete rows back to back and keeps NV * kRowsPerStep 16-byte
// loads in flight per thread.
template <int NV>
__global__ void __launch_bounds__(kThreads) relayout_rows_kernel(const uint16_t* __restrict__ src,
                                                                 uint16_t* __restrict__ dst, int64_t row_stride,
                                                                 int64_t rows, int n_heads, int head_dim,
                                                                 int heads_per_group, int pack) {
    const int vec_per_head = head_dim >> 3;
    const int vec_per_row = n_heads * vec_per_head;
    const int64_t grp_row = (int64_t)heads_per_group * head_dim;
    const int64_t group_elems = rows * grp_row;
    const int64_t row_step = pack ? row_stride : grp_row;
    const int64_t dst_step = pack ? grp_row : row_stride;
    int64_t soff[NV], doff[NV];
    bool ok[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        const int v = threadIdx.x + j * kThreads;
        ok[j] = v < vec_per_row;
        const int vc = ok[j] ? v : 0;
        const int h = vc / vec_per_head;
        const int e = vc - h * vec_per_head;
        const int g = h / heads_per_group;
        const int hl = h - g * heads_per_group;
        const int64_t row_col = (int64_t)vc * 8;
        const int64_t grp_col = g * group_elems + (int64_t)hl * head_dim + e * 8;
        soff[j] = pack ? row_col : grp_col;
        doff[j] = pack ? grp_col : row_col;
    }
    const int64_t r0 = rows * (int64_t)blockIdx.x / gridDim.x;
    const int64_t r1 = rows * (int64_t)(blockIdx.x + 1) / gridDim.x;
    grid_dep_wait();
    int64_t r = r0;
    for (; r + kRowsPerStep <= r1; r += kRowsPerStep) {
        Vec8 t[kRowsPerStep][NV];
#pragma unroll
        for (int k = 0; k < kRowsPerStep; ++k)
#pragma unroll
            for (int j = 0; j < NV; ++j)
                if (ok[j]) t[k][j] = ld_ro(src + soff[j] + (r + k) * row_step);
#pragma unroll
        for (int k = 0; k < kRowsPerStep; ++k)
#pragma unroll
            for (int j = 0; j < NV; ++j)
                if (ok[j]) st_vec(dst + doff[j] + (r + k) * dst_step, t[k][j]);
    }
    for (; r < r1; ++r)
#pragma unroll
        for (int j = 0; j < NV; ++j)
            if (ok[j]) st_vec(dst + doff[j] + r * dst_step, ld_ro(src + soff[j] + r * row_step));
}

}  // namespace

cudaError_t launch_ulysses_relayout(const uint16_t* src, uint16_t* dst, int64_t row_stride, int64_t rows,
                                    int n_heads, int head_dim, int groups, bool pack, cudaStream_t stream) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    const int nv = (n_heads * (head_dim / 8) + kThreads - 1) / kThreads;
    using Kern = void (*)(const uint16_t*, uint16_t*, int64_t, int64_t, int, int, int, int);
    Kern k = relayout_kernel;  // more than 8192 values per row
    if (nv == 1) k = relayout_rows_kernel<1>;
    else if (nv == 2) k = relayout_rows_kernel<2>;
    else if (nv == 3) k = relayout_rows_kernel<3>;
    else if (nv == 4) k = relayout_rows_kernel<4>;
    const int per_sm = blocks_per_sm(reinterpret_cast<const void*>(k), kThreads, 0);
    if (per_sm <= 0) return cudaErrorInvalidConfiguration;
    // One CTA per kRowsPerCta rows, balanced over the SMs by the hardware block
    // scheduler, once that is more CTAs than one resident wave; the static
    // split of one persistent run per CTA left SMs idle at the end.  Measured
    // (40 x 128 heads, 75,600 rows, 8 ranks): 92% -> 100% of the copy
    // bandwidth; 24 x 128 and 8 x 128: 88% -> 97%.
    int64_t grid = (int64_t)per_sm * di.sm_count;
    const int64_t tiles = (rows + kRowsPerCta - 1) / kRowsPerCta;
    if (tiles > grid) grid = tiles;
    if (grid > (1 << 24)) grid = 1 << 24;  // the row split covers any grid; keeps rows * blockIdx in range
    if (grid > rows) grid = rows;
    return launch_kernel(k, (unsigned)grid, kThreads, 0, stream, src, dst, row_stride, rows,
                         n_heads, head_dim, n_heads / groups, pack ? 1 : 0);
}

}  // namespace tfk
