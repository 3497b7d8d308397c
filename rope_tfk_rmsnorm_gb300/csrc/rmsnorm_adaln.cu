// rmsnorm_adaln.cu - RMSNorm fused with indexed AdaLN modulation.
//
// y[t,j] = bf16( x[t,j] * rsqrt(mean_j x[t,:]^2 + eps) * w[j] * (1 + scale[m,j]) + shift[m,j] ),
// m = mod_idx[t].  TeleFuser PR #38, section 2: RMSNorm fused with the
// per-token indexed AdaLN modulation; TeleFuser PR #23, section Changes
// Made: the indexed-modulation kernel.
//
// Three kernels, chosen by hidden alone (so a row's output bits never depend
// on the rows of the call):
// - rmsnorm_adaln_kernel, one CTA per row (below);
// - the same kernel in pairs (kPair): a cluster of two CTAs per row, each with
//   half the columns, for rows wider than 17408;
// - rmsnorm_adaln_warp_kernel, one warp per row with the modulation staged in
//   shared memory, for the widths where the CTA shape keeps rows unsorted
//   (see "one warp per row" below).
//
// Design of the CTA-per-row kernel (HBM-bound: 2 bytes read + 2 bytes written
// per element):
// - Persistent CTAs, each owning a contiguous run of rows, so the modulation
//   index changes rarely inside a CTA in the packed video+audio layout.
// - Each thread owns the same 8*V columns of every row.  The norm weight for
//   those columns lives in registers for the whole kernel, and the shift and
//   (1 + scale) of the current modulation row are cached in registers and
//   re-read only when mod_idx changes (two cached rows when V == 1, i.e.
//   hidden < 512, so a per-token choice between two rows costs no reload).
//   In steady state the fp32 parameters cost no memory traffic at all.
// - Activation rows are staged through a shared-memory ring with cp.async
//   (16 B per thread, L1 bypassed), `stages - 1` rows ahead, so many rows are
//   in flight per SM without holding them in registers.  A thread only reads
//   back the slots it copied itself, so no barrier guards the ring.
// - Sum of squares: fp32 per thread, warp shuffle, then one barrier per row
//   through a double-buffered array of per-warp partials.
#include "../../include/tfk.h"
#include "common.cuh"
#include "kernels.h"

namespace tfk {
namespace {

constexpr int kMaxThreads = 512;
constexpr int kMaxThreadsV1 = 384;
// Rows per CTA: one persistent run per resident CTA, unless such a run would
// exceed kChunkMinRun rows; then chunks of kRowsPerCta rows (kRowsPerCtaWide
// for rows of 16 KB and more) that the hardware block scheduler balances over
// the SMs.  Measured on the GB300: chunks of 24 gain 1.5-2% at 56,320-75,600
// rows (runs of 93-166 rows), while at 30,358 rows of 3072 (runs of 40) the
// persistent split is 4% faster.  Chunks of 16 rather than 24 (fraction of
// the copy bandwidth, event-timed): 75,600 x 5120 0.962 -> 0.974, 56,320 x
// 4096 0.922 -> 0.929, but 20,000 x 8192 0.758 -> 0.734 (there each chunk
// also reloads 96 KB of modulation), so wide rows keep 24; 12 and 32 rows
// measured no better than these.
#ifndef TFK_A1_CHUNK_MIN_RUN
#define TFK_A1_CHUNK_MIN_RUN 64
#endif
constexpr int64_t kRowsPerCta = 16;
constexpr int64_t kRowsPerCtaWide = 24;
template <int V, bool kExact>
constexpr bool kSortRows = V == 2 || (V == 4 && kExact);
constexpr int kSortRun = 64;  // at most 256: row positions are stored as bytes
constexpr int64_t kChunkMinRun = TFK_A1_CHUNK_MIN_RUN;

// Combined modulation of the columns a thread owns for modulation row m:
//   mul = w * (1 + scale[m]),  add = shift[m]
// so that y = x * inv_rms * mul + add (one fp32 rounding of w * (1 + scale)
// more than the literal formula; far below the bf16 rounding of y).
template <int V>
__device__ __forceinline__ void load_mod_row(const AdalnArgs& a, int m, const int (&col)[V],
                                             const bool (&ok)[V], float (&mul)[V][8], float (&add)[V][8]) {
    const float* srow = a.shift + (int64_t)m * a.hidden;
    const float* crow = a.scale + (int64_t)m * a.hidden;
#pragma unroll
    for (int i = 0; i < V; ++i) {
        if (ok[i]) {
            const float4 s0 = ld_f4(srow + col[i] * 8), s1 = ld_f4(srow + col[i] * 8 + 4);
            const float4 c0 = ld_f4(crow + col[i] * 8), c1 = ld_f4(crow + col[i] * 8 + 4);
            const float4 w0 = ld_f4(a.weight + col[i] * 8), w1 = ld_f4(a.weight + col[i] * 8 + 4);
            add[i][0] = s0.x; add[i][1] = s0.y; add[i][2] = s0.z; add[i][3] = s0.w;
            add[i][4] = s1.x; add[i][5] = s1.y; add[i][6] = s1.z; add[i][7] = s1.w;
            mul[i][0] = w0.x * (1.0f + c0.x); mul[i][1] = w0.y * (1.0f + c0.y);
            mul[i][2] = w0.z * (1.0f + c0.z); mul[i][3] = w0.w * (1.0f + c0.w);
            mul[i][4] = w1.x * (1.0f + c1.x); mul[i][5] = w1.y * (1.0f + c1.y);
            mul[i][6] = w1.z * (1.0f + c1.z); mul[i][7] = w1.w * (1.0f + c1.w);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) { mul[i][e] = 0.f; add[i][e] = 0.f; }
        }
    }
}

// One or two vectors per thread (hidden < 4096) run at least two CTAs per
// SM, so that their per-row reductions and barriers overlap: one vector per
// thread (two cached modulation rows) within 85 registers, two vectors within
// 64; wider rows get the full register file.
// MAXT: most threads per CTA of this instantiation.  kExact: every thread
// owns V whole vectors (8 * V * threads == hidden: hidden a multiple of 512
// for V = 2, of 1024 for V = 4), so no bounds predicates.  Two vectors in at
// most 256 threads get 80 registers when exact: with 64 the compiler re-read
// thread indices and kernel parameters inside the row loop.  Measured
// against 64 registers with predicates: +7 points at hidden 2048, +3 at
// 3072 x 8192 rows, even at 3072 x 30358; four exact vectors +1.5 points at
// 4096 and 5120.
template <int V, int MAXT, bool kExact>
constexpr int kMinBlocks = V == 1 ? 2 : (V == 2 ? (MAXT <= 256 && kExact ? 3 : 2 * (512 / MAXT))
                                                : (V == 3 ? 3 : 1));

// kPair: a cluster of two CTAs shares each row, for rows too wide for one CTA
// to hold the modulation of its columns in registers (hidden > 16384).  CTA c
// of the pair takes the columns of vectors [c * half, ...) (half = the first
// ceil(nvec / 2) vectors), both run the pair's rows in the same order, and
// per row each adds the other's partial sum of squares, exchanged through
// distributed shared memory with one cluster barrier; both then form the same
// total, partial(CTA 0) + partial(CTA 1).
template <int V, int MAXT, bool kExact, bool kPair = false>
__global__ void __launch_bounds__(MAXT, (kMinBlocks<V, MAXT, kExact>))
rmsnorm_adaln_kernel(const AdalnArgs args, const int stages) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Vec8* ring = reinterpret_cast<Vec8*>(smem_raw);  // [stages][nvec]
    __shared__ float partial[2][32];
    __shared__ float xchg[2][2];  // [row parity][CTA of the pair]: partial sums (kPair)
    grid_dep_wait();

    const unsigned crank = kPair ? cluster_ctarank() : 0u;
    const int half = ((args.hidden >> 3) + 1) >> 1;
    // vectors of this CTA's columns
    const int nvec = !kPair ? args.hidden >> 3 : (crank ? (args.hidden >> 3) - half : half);
    const unsigned unit = kPair ? blockIdx.x >> 1 : blockIdx.x;
    const unsigned units = kPair ? gridDim.x >> 1 : gridDim.x;
    AdalnArgs half_args = args;  // kPair: the arguments moved to this CTA's columns
    if constexpr (kPair) {
        const int cbase = crank ? half : 0;
        half_args.x += cbase * 8;
        half_args.y += cbase * 8;
        half_args.weight += cbase * 8;
        half_args.shift += cbase * 8;
        half_args.scale += cbase * 8;
    }
    const AdalnArgs& a = kPair ? half_args : args;
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = (nt + 31) >> 5;
    const float inv_hidden = 1.0f / (float)a.hidden;

    const int64_t r0 = a.rows * (int64_t)unit / units;
    const int64_t r1 = a.rows * (int64_t)(unit + 1) / units;
    const int nrows = (int)(r1 - r0);

    int col[V];
    bool ok[V];
#pragma unroll
    for (int i = 0; i < V; ++i) {
        col[i] = tid + i * nt;
        ok[i] = kExact || col[i] < nvec;
    }

    // Two vectors, and four whole vectors, per thread: the CTA's rows in order
    // of modulation index (stable), so that a run whose tokens alternate
    // between modulation rows reloads each row about once instead of on every
    // switch; for constant or sorted indices the order is the identity.  Every
    // row is still read and written once, at its own address.  Runs are at
    // most 64 rows at the launch shapes; a longer one keeps its natural order.
    // Measured with per-token coin flips between two modulation rows: 5120
    // 67% -> 88% of the copy bandwidth, 2048 66% -> 81%, 1024 70% -> 77%;
    // constant indices 5120 +0.3, per-frame +1.5, 2048 -1.3.  The
    // three-vector and the predicated four-vector instantiations keep the
    // natural order: there the extra state spilled (constant indices -8 and
    // -3.7 points).
    __shared__ int s_key[kSortRows<V, kExact> ? kSortRun : 1];
    __shared__ unsigned char s_order[kSortRows<V, kExact> ? kSortRun : 1];
    bool sorted = false;
    if constexpr (kSortRows<V, kExact>) {
        sorted = nrows > 1 && nrows <= kSortRun;  // uniform over the CTA
        if (sorted) {
            for (int j = tid; j < nrows; j += nt) s_key[j] = __ldg(a.mod_idx + r0 + j);
            __syncthreads();
            for (int j = tid; j < nrows; j += nt) {
                const int kj = s_key[j];
                int rank = 0;
                for (int u = 0; u < nrows; ++u) {
                    const int ku = s_key[u];
                    rank += (ku < kj) | ((ku == kj) & (u < j));
                }
                s_order[rank] = (unsigned char)j;
            }
            __syncthreads();
        }
    }
    auto row_at = [&](int i) -> int { return sorted ? (int)s_order[i] : i; };
    auto key_at = [&](int i) -> int { return sorted ? s_key[s_order[i]] : __ldg(a.mod_idx + r0 + i); };

    if (nrows > 0) {  // uniform over the CTA
        // Prologue: rows 0 .. stages-2 of this CTA's run go in flight.
        for (int s = 0; s < stages - 1; ++s) {
            if (s < nrows) {
                const uint16_t* src = a.x + (r0 + row_at(s)) * a.x_stride;
                Vec8* dst = ring + (int64_t)s * nvec;
#pragma unroll
                for (int i = 0; i < V; ++i)
                    if (ok[i]) cp_async16(dst + col[i], src + col[i] * 8);
            }
            cp_async_commit();
        }

        // The first row's modulation is fetched while the prologue rows are in
        // flight, not after the first row has arrived.
        float mul[V][8], add[V][8];
        float mul2[1][8], add2[1][8];  // second cached row (used when V == 1)
        int m_cur = key_at(0), m_alt = -1;
        load_mod_row<V>(a, m_cur, col, ok, mul, add);
        int m_next = m_cur;
        int stage_rd = 0, stage_wr = stages - 1;

        for (int it = 0; it < nrows; ++it) {
            const int64_t r = r0 + row_at(it);
            {   // keep stages-1 rows in flight
                const int ahead = it + stages - 1;
                if (ahead < nrows) {
                    const uint16_t* src = a.x + (r0 + row_at(ahead)) * a.x_stride;
                    Vec8* dst = ring + (int64_t)stage_wr * nvec;
#pragma unroll
                    for (int i = 0; i < V; ++i)
                        if (ok[i]) cp_async16(dst + col[i], src + col[i] * 8);
                }
                cp_async_commit();
                stage_wr = stage_wr + 1 == stages ? 0 : stage_wr + 1;
            }
            const int m = m_next;
            if (it + 1 < nrows) m_next = key_at(it + 1);
            cp_async_wait_dyn(stages - 1);

            const Vec8* cur = ring + (int64_t)stage_rd * nvec;
            stage_rd = stage_rd + 1 == stages ? 0 : stage_rd + 1;
            Vec8 xv[V];
            float ss0 = 0.f, ss1 = 0.f;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                if (ok[i]) {
                    xv[i] = ld_smem_vec(cur + col[i]);
                } else {
                    xv[i].w[0] = xv[i].w[1] = xv[i].w[2] = xv[i].w[3] = 0u;
                }
                float f[8];
                unpack8(xv[i], f);
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    ss0 = fmaf(f[e], f[e], ss0);
                    ss1 = fmaf(f[e + 1], f[e + 1], ss1);
                }
            }
            float ss = warp_sum(ss0 + ss1);
            if (lane == 0) partial[it & 1][warp] = ss;

            if (m != m_cur) {  // uniform over the CTA; the loads overlap the barrier below
                if constexpr (V == 1) {
                    if (m == m_alt) {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const float tm = mul[0][e], ta = add[0][e];
                            mul[0][e] = mul2[0][e]; add[0][e] = add2[0][e];
                            mul2[0][e] = tm; add2[0][e] = ta;
                        }
                        m_alt = m_cur;
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) { mul2[0][e] = mul[0][e]; add2[0][e] = add[0][e]; }
                        m_alt = m_cur;
                        load_mod_row<V>(a, m, col, ok, mul, add);
                    }
                } else {
                    load_mod_row<V>(a, m, col, ok, mul, add);
                }
                m_cur = m;
            }

            __syncthreads();
            float total = warp_sum(lane < nwarps ? partial[it & 1][lane] : 0.f);
            if constexpr (kPair) {
                if (tid == 0) {
                    xchg[it & 1][crank] = total;
                    st_peer_f32(&xchg[it & 1][crank], crank ^ 1u, total);
                }
                cluster_sync();  // both partials of this row are in both CTAs
                total = xchg[it & 1][0] + xchg[it & 1][1];
            }
            const float inv_rms = rsqrtf(total * inv_hidden + a.eps);

            uint16_t* dst = a.y + r * a.y_stride;
#pragma unroll
            for (int i = 0; i < V; ++i) {
                if (ok[i]) {
                    float f[8], o[8];
                    unpack8(xv[i], f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = fmaf(f[e] * inv_rms, mul[i][e], add[i][e]);
                    st_vec(dst + col[i] * 8, pack8(o));
                }
            }
        }
        cp_async_wait<0>();
    }  // nrows > 0

    // Fixed-valid mode: this CTA's share of the padded tail is written +0.0
    // in the same launch (stores only; the tail of x is never read).
    const int64_t tail = a.padded_rows - a.rows;
    if (tail > 0) {
        const int64_t z0 = a.rows + tail * (int64_t)unit / units;
        const int64_t z1 = a.rows + tail * (int64_t)(unit + 1) / units;
        Vec8 zero;
        zero.w[0] = zero.w[1] = zero.w[2] = zero.w[3] = 0u;
        for (int64_t r = z0; r < z1; ++r) {
            uint16_t* dst = a.y + r * a.y_stride;
#pragma unroll
            for (int i = 0; i < V; ++i)
                if (ok[i]) st_vec(dst + col[i] * 8, zero);
        }
    }
    // No CTA of a pair leaves while the other may still write to its shared memory.
    if constexpr (kPair) cluster_sync();
}

// ---- one warp per row --------------------------------------------------------
//
// A warp owns whole rows: lane l holds vectors l, l+32, ... of the row in
// registers (VPL per lane), the sum of squares is one warp shuffle, and no
// barrier or shared-memory exchange sits in the row loop at all.  A CTA owns a
// contiguous run of rows and hands them to its warps in turn.  The modulation
// of the rows it uses, mul = w * (1 + scale[m]) and add = shift[m], is
// precombined into shared memory once, in four 16-byte planes per vector so
// that the lanes of a warp read consecutive 16-byte words (no bank conflicts):
//   tab[slot][plane][v], plane 0/1 = mul of elements 0-3 / 4-7, plane 2/3 = add.
// Modulation row m may only use slot m % slots.  When every modulation row
// has a slot (n_mod <= slots, as in every workload here), the CTA stages them
// all in one pass without reading the indices first.  Otherwise, in a pass,
// each slot holds the smallest m of the CTA's not yet computed rows that maps
// to it, and the rows whose m is staged are computed; passes repeat until
// every row is done (one pass when the CTA's rows use at most `slots` rows).
// A row's arithmetic never depends on the slot, the pass or the launch shape,
// so the output bits do not depend on how the rows are split between CTAs or
// between calls.
constexpr int kWarpMaxSlots = 64;
constexpr int kNoRow = 0x7FFFFFFF;
// Dynamic row hand-out (with the caller's workspace): kSchedGroups row
// counters kSchedStride 64-bit words (256 bytes) apart, then the count of
// finished CTAs at word kDoneWord.
constexpr int kSchedGroups = 4;
constexpr int kSchedStride = 32;
constexpr int kDoneWord = 8 * kSchedStride;
static_assert(kSchedGroups * kSchedStride <= kDoneWord, "counters overlap the completion count");
static_assert((kDoneWord + 1) * 8 <= TFK_RMSNORM_WORKSPACE_BYTES, "workspace too small");

// Threads per CTA (one CTA per SM): the register budget of a thread is
// 65536 / threads, and one row takes 4 * VPL registers of a lane.  Measured at
// 12 vectors per lane: 768 threads and 640 equal; three CTAs of 256 or two of
// 384 per SM 1-4 points lower.
template <int VPL>
constexpr int kWarpThreads = VPL <= 4 ? 1024 : (VPL <= 12 ? 768 : (VPL <= 16 ? 640 : (VPL <= 20 ? 512 : 448)));

// RMSNorm + modulation of one row held in registers, stored to y.
// t: the row's modulation slot in the shared table, offset by the lane.
template <int VPL, bool kExact>
__device__ __forceinline__ void warp_row_out(const AdalnArgs& a, int64_t row, int lane, int nvec, float inv_hidden,
                                             const float4* t, const Vec8 (&xv)[VPL]) {
    float ss0 = 0.f, ss1 = 0.f;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float lo = __uint_as_float(xv[j].w[k] << 16), hi = __uint_as_float(xv[j].w[k] & 0xFFFF0000u);
            ss0 = fmaf(lo, lo, ss0);
            ss1 = fmaf(hi, hi, ss1);
        }
    }
    const float inv_rms = rsqrtf(warp_sum(ss0 + ss1) * inv_hidden + a.eps);
    const f32x2 r2 = f2_make(inv_rms, inv_rms);
    // The output pass widens the bf16 words again, with byte permutes whose
    // selectors carry a dependence on inv_rms (bit 16 and up of a selector is
    // ignored, so the values are those of the plain widening).  Without it the
    // compiler widened every word ahead, during the shuffles, and the widened
    // row no longer fit in the register budget (spills).
    const unsigned dep = (__float_as_uint(inv_rms) >> 31) << 16;
    const unsigned sel_lo = 0x1044u | dep, sel_hi = 0x3244u | dep;
    uint16_t* dst = a.y + row * a.y_stride + lane * 8;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
        if (!(kExact || j * 32 + lane < nvec)) continue;
        const float4 m0 = t[j * 32], m1 = t[nvec + j * 32];
        const float4 b0 = t[2 * nvec + j * 32], b1 = t[3 * nvec + j * 32];
        f32x2 xw[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            xw[k] = f2_make(__uint_as_float(__byte_perm(xv[j].w[k], 0u, sel_lo)),
                            __uint_as_float(__byte_perm(xv[j].w[k], 0u, sel_hi)));
        Vec8 o;
        o.w[0] = f2_to_bf2(f2_fma(f2_mul(xw[0], r2), f2_make(m0.x, m0.y), f2_make(b0.x, b0.y)));
        o.w[1] = f2_to_bf2(f2_fma(f2_mul(xw[1], r2), f2_make(m0.z, m0.w), f2_make(b0.z, b0.w)));
        o.w[2] = f2_to_bf2(f2_fma(f2_mul(xw[2], r2), f2_make(m1.x, m1.y), f2_make(b1.x, b1.y)));
        o.w[3] = f2_to_bf2(f2_fma(f2_mul(xw[3], r2), f2_make(m1.z, m1.w), f2_make(b1.z, b1.w)));
        st_vec(dst + j * 256, o);
    }
}

template <int VPL, bool kExact>
__global__ void __launch_bounds__(kWarpThreads<VPL>, 1)
rmsnorm_adaln_warp_kernel(const AdalnArgs a, const int slots, const int n_mod) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    float4* tab = reinterpret_cast<float4*>(smem_raw);  // [slots][4][nvec]
    __shared__ int slot_m[kWarpMaxSlots];                // staged m per slot in this pass (kNoRow: none)
    __shared__ int done_m[kWarpMaxSlots];                // rows with m <= done_m[m % slots] are computed
    __shared__ int claimed_list[kWarpMaxSlots];
    __shared__ int n_claimed;
    __shared__ int more_passes;

    const int nvec = a.hidden >> 3;
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = nt >> 5;
    const float inv_hidden = 1.0f / (float)a.hidden;
    const int64_t r0 = a.rows * (int64_t)blockIdx.x / gridDim.x;
    const int64_t r1 = a.rows * (int64_t)(blockIdx.x + 1) / gridDim.x;

    for (int s = tid; s < slots; s += nt) done_m[s] = -1;
    grid_dep_wait();

    // The next row of this warp after `r` whose modulation row is staged in
    // this pass (r1 if none), and its slot.
    auto next_staged = [&](int64_t r, int& slot) -> int64_t {
        for (r += nwarps; r < r1; r += nwarps) {
            const int m = __ldg(a.mod_idx + r);
            slot = m % slots;
            if (slot_m[slot] == m) return r;
        }
        return r1;
    };

    // With a workspace and every modulation row staged, rows are handed out
    // as warps become free (uniform over the launch).  The rows are dealt to
    // kSchedGroups groups of CTAs (CTA b in group b % groups), group g taking
    // rows g, g + groups, g + 2 * groups, ...; a warp claims the next row of
    // its group with one atomic on the group's counter.  Measured (fraction of
    // the copy bandwidth, event-timed) against rows split up front: 30,358 x
    // 3072 0.79 -> 0.85, 75,600 x 3072 0.88 -> 0.95, 30,000 x 4352 0.81 ->
    // 0.88 (smaller calls get no counters: kHandOutMinBytesPerSm).  One
    // counter for all SMs queued the claims at 75,600 x 3072 (0.59); two
    // counters 0.89, four and eight 0.94-0.95.  Claiming one row ahead, or
    // several rows per claim in shrinking chunks, measured 1-6 points lower.
    const bool dynamic = a.sched != nullptr && slots >= n_mod;
    const int groups = gridDim.x < (unsigned)kSchedGroups ? (int)gridDim.x : kSchedGroups;
    const int grp = (int)(blockIdx.x % (unsigned)groups);
    unsigned long long* gctr = dynamic ? a.sched + (int64_t)grp * kSchedStride : nullptr;
    const int64_t grows = (a.rows - grp + groups - 1) / groups;  // rows of this group
    for (;;) {
        bool last_pass = true;
        if (slots >= n_mod) {
            // Every modulation row has a slot of its own (m % slots == m): one
            // pass that stages all of them, without reading the indices first.
            for (int s = tid; s < slots; s += nt) {
                slot_m[s] = s;
                claimed_list[s] = s;
            }
            if (tid == 0) n_claimed = slots;
            __syncthreads();
        } else {
            for (int s = tid; s < slots; s += nt) slot_m[s] = kNoRow;
            if (tid == 0) more_passes = 0;
            __syncthreads();
#pragma unroll 1
            for (int64_t i = r0 + tid; i < r1; i += nt) {
                const int m = __ldg(a.mod_idx + i);
                if (m > done_m[m % slots]) atomicMin(&slot_m[m % slots], m);
            }
            __syncthreads();
            // A row whose modulation row lost its slot needs another pass.
            bool claimed = false, left = false;
            for (int s = tid; s < slots; s += nt) claimed |= slot_m[s] != kNoRow;
#pragma unroll 1
            for (int64_t i = r0 + tid; i < r1; i += nt) {
                const int m = __ldg(a.mod_idx + i);
                left |= m > done_m[m % slots] && slot_m[m % slots] != m;
            }
            if (left) more_passes = 1;
            if (tid == 0) {
                int n = 0;
                for (int s = 0; s < slots; ++s)
                    if (slot_m[s] != kNoRow) claimed_list[n++] = s;
                n_claimed = n;
            }
            if (!__syncthreads_or(claimed)) break;  // uniform: every row is computed
            last_pass = more_passes == 0;
        }


        // The claimed modulation rows, staged as one flat loop over
        // (slot, vector) so that all their loads are in flight together.
        // Building the table costs 1.2-3 us per launch (measured by leaving it
        // out: 8,192 x 3072 26.0 -> 24.3 us, 30,000 x 6144 120 -> 117 us).
        // Measured equal or slower: shift and scale copied into the table
        // with cp.async and combined in place (+4.5 us at 8,192 x 3072), w
        // read once per half-vector for all slots, the warp's first row issued
        // or prefetched into L2 before the table, and a first row per warp
        // assigned without a claim.
        const int items = n_claimed * nvec;
#pragma unroll 2
        for (int it = tid; it < items; it += nt) {
            const int s = claimed_list[it / nvec], v = it - (it / nvec) * nvec;
            const int m = slot_m[s];
            const float* srow = a.shift + (int64_t)m * a.hidden;
            const float* crow = a.scale + (int64_t)m * a.hidden;
            float4* t = tab + (int64_t)s * 4 * nvec;
            const float4 w0 = ld_f4(a.weight + v * 8), w1 = ld_f4(a.weight + v * 8 + 4);
            const float4 c0 = ld_f4(crow + v * 8), c1 = ld_f4(crow + v * 8 + 4);
            const float4 b0 = ld_f4(srow + v * 8), b1 = ld_f4(srow + v * 8 + 4);
            t[v] = make_float4(w0.x * (1.0f + c0.x), w0.y * (1.0f + c0.y), w0.z * (1.0f + c0.z), w0.w * (1.0f + c0.w));
            t[nvec + v] = make_float4(w1.x * (1.0f + c1.x), w1.y * (1.0f + c1.y), w1.z * (1.0f + c1.z),
                                      w1.w * (1.0f + c1.w));
            t[2 * nvec + v] = b0;
            t[3 * nvec + v] = b1;
        }
        __syncthreads();

        // The next row of this warp after `r` (and its slot): with dynamic
        // hand-out the next row of its group's counter (slot == m, since every
        // row has its own slot); otherwise the next staged row of the CTA's
        // run.  `rend` once there is none.
        const int64_t rend = dynamic ? a.rows : r1;
        auto advance = [&](int64_t r, int& slot) -> int64_t {
            if (dynamic) {
                unsigned long long got = 0;
                if (lane == 0) got = atomicAdd(gctr, 1ull);
                got = __shfl_sync(0xFFFFFFFFu, got, 0);
                if ((int64_t)got >= grows) return rend;
                const int64_t row = (int64_t)got * groups + grp;
                slot = __ldg(a.mod_idx + row);
                return row;
            }
            return next_staged(r, slot);
        };
        int sa = 0;
#pragma unroll 1
        for (int64_t r = advance(r0 + warp - nwarps, sa); r < rend; r = advance(r, sa)) {
            Vec8 xv[VPL];
            const uint16_t* src = a.x + r * a.x_stride + lane * 8;
#pragma unroll
            for (int j = 0; j < VPL; ++j) {
                if (kExact || j * 32 + lane < nvec) {
                    xv[j] = ld_ro(src + j * 256);
                } else {
                    xv[j].w[0] = xv[j].w[1] = xv[j].w[2] = xv[j].w[3] = 0u;
                }
            }
            warp_row_out<VPL, kExact>(a, r, lane, nvec, inv_hidden, tab + (int64_t)sa * 4 * nvec + lane, xv);
        }
        if (last_pass) break;  // uniform: no barrier needed after the last pass
        __syncthreads();  // the next pass rewrites slot_m and the table
        for (int s = tid; s < slots; s += nt)
            if (slot_m[s] != kNoRow) done_m[s] = slot_m[s];
    }

    if (dynamic) {
        // The last CTA to finish claiming returns the counters to zero for the
        // next call (no CTA claims again once it has counted itself finished).
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            unsigned long long* done = a.sched + kDoneWord;
            if (atomicAdd(done, 1ull) == (unsigned long long)gridDim.x - 1) {
                for (int g = 0; g < kSchedGroups; ++g) atomicExch(a.sched + (int64_t)g * kSchedStride, 0ull);
                atomicExch(done, 0ull);
            }
        }
    }

    // Fixed-valid mode: this CTA's share of the padded tail is written +0.0.
    const int64_t tail = a.padded_rows - a.rows;
    if (tail > 0) {
        const int64_t z0 = a.rows + tail * (int64_t)blockIdx.x / gridDim.x;
        const int64_t z1 = a.rows + tail * (int64_t)(blockIdx.x + 1) / gridDim.x;
        Vec8 zero;
        zero.w[0] = zero.w[1] = zero.w[2] = zero.w[3] = 0u;
        for (int64_t z = z0 + warp; z < z1; z += nwarps) {
            uint16_t* dst = a.y + z * a.y_stride + lane * 8;
#pragma unroll
            for (int j = 0; j < VPL; ++j)
                if (kExact || j * 32 + lane < nvec) st_vec(dst + j * 256, zero);
        }
    }
}

// Two vectors per thread from hidden 512 on, four from 4096 (128-160
// threads, a barrier over 4-5 warps: +2% at hidden 4096 and 5120 over two),
// eight beyond 16384.  Short rows are issue-bound rather than memory-bound:
// the per-row loop, ring wait, two shuffle reductions and barrier are paid
// for 8 elements per thread with one vector.  Two vectors per thread instead
// of one measured 58% -> 79-83% of the copy bandwidth at hidden 512-1536
// (constant index; 54% -> 66-68% with a per-token coin flip, despite losing
// the second cached modulation row), and let four or more 64-register CTAs
// share an SM.  One vector per thread is left for hidden < 512.  Hidden
// 6144-8192 goes back to two vectors: four would take ~120 registers for
// 192-256 threads, i.e. two CTAs of 6-8 warps per SM (measured 74% -> 78% at
// 6144, +1% at 8192; at 4096 and 5120 four vectors stay ahead).  Beyond
// 16384 eight vectors do not fit in 128 registers and spill (~40-47%).
// Hidden a multiple of 768 from 1536 to 6144 takes three whole vectors per
// thread (64-256 threads, 80 registers): the per-row overhead is spread over
// 24 elements and the barrier spans fewer warps.  Measured against the
// shapes above: 5376 68% -> 88%, 6144 78% -> 86%, 4608 83% -> 88%,
// 1536-2304 +4.5 points, 3072 +1.
#ifndef TFK_A1_MIN_V
#define TFK_A1_MIN_V 2
#endif
#ifndef TFK_A1_V2_FROM_NVEC
#define TFK_A1_V2_FROM_NVEC 64
#endif
#ifndef TFK_A1_V4_FROM_NVEC
#define TFK_A1_V4_FROM_NVEC 512
#endif
bool choose_shape(int hidden, int* v, int* threads) {
    const int nvec = hidden / 8;
    int first = nvec >= TFK_A1_V4_FROM_NVEC ? 4 : (nvec >= TFK_A1_V2_FROM_NVEC ? TFK_A1_MIN_V : 1);
    if (nvec >= 768 && nvec <= 1024) first = 2;  // hidden 6144-8192: 384-512 threads of 64 registers
    if (nvec % 96 == 0 && nvec / 3 <= 256 && nvec >= 192) {  // three whole vectors per thread
        *v = 3;
        *threads = nvec / 3;
        return true;
    }
    for (int cand = first; cand <= 8; cand *= 2) {
        const int t = (nvec + cand - 1) / cand;
        if (t <= (cand == 1 ? kMaxThreadsV1 : kMaxThreads)) {
            *v = cand;
            *threads = (t + 31) / 32 * 32;
            return true;
        }
    }
    return false;
}

template <int V, int MAXT, bool kExact>
cudaError_t launch_v(const AdalnArgs& a, int threads, cudaStream_t stream) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    const int row_bytes = (a.hidden / 8) * 16;
    const void* fn = reinterpret_cast<const void*>(&rmsnorm_adaln_kernel<V, MAXT, kExact>);
    const int by_regs = blocks_per_sm(fn, threads, 0);
    if (by_regs <= 0) return cudaErrorInvalidConfiguration;
    // Rows of 16 KB and more (hidden >= 8192) keep 80 KB in flight per SM
    // instead of 112: measured +1.5-2 points at hidden 12288 and 16384 (the
    // ring then takes fewer of the SM's 228 KB of shared memory).
    const int stages = pick_stages(by_regs, row_bytes, 0, row_bytes >= 16384 ? 80 * 1024 : kInflightPerSm);
    const size_t smem = (size_t)stages * row_bytes;
    const int per_sm = blocks_per_sm(fn, threads, smem);
    if (per_sm <= 0) return cudaErrorInvalidConfiguration;
    int64_t grid = (int64_t)per_sm * di.sm_count;
    const int64_t work = a.rows > a.padded_rows - a.rows ? a.rows : a.padded_rows - a.rows;
    {  // fixed-size chunks instead of long persistent runs
        const int64_t per = row_bytes >= 16384 ? kRowsPerCtaWide : kRowsPerCta;
        const int64_t chunks = (work + per - 1) / per;
        if (chunks > grid && work >= kChunkMinRun * grid) grid = chunks;
    }
    if (grid > (1 << 24)) grid = 1 << 24;  // the row split covers any grid; keeps rows * blockIdx in range
    if (grid > work) grid = work;
    if (grid < 1) return cudaSuccess;
    return launch_kernel(rmsnorm_adaln_kernel<V, MAXT, kExact>, (unsigned)grid, threads, smem, stream, a, stages);
}

// The warp-per-row kernel takes the widths whose CTA-per-row shape keeps the
// rows in their natural order (three whole vectors per thread, or four with
// a ragged last thread), from 256 to 5120.  There a per-token change of
// modulation row reloads the CTA's register-cached modulation on every
// switch, while the warp kernel reads any staged row from shared memory.
// Measured on the GB300 (event-timed launches, fraction of the measured copy
// bandwidth, CTA kernel -> warp kernel):
//   hidden 3072,  8,192 rows, 4 rows by modality and per-token coin flip: 0.48 -> 0.58
//   hidden 3072, 30,358 rows, per-token coin flip between 2 rows:        0.64 -> 0.78
//   hidden 4352, 30,000 rows, per-token coin flip:                        0.55 -> 0.81
// and with long constant runs of one row the CTA kernel stays ahead by 1-3
// points at these widths (3072 x 30,358: 0.81 vs 0.78), by 7-15 at the
// widths that keep it (four whole vectors: 5120 0.96 vs 0.89, 4096 0.92
// vs 0.78), where its row sort already handles alternating rows.
#ifndef TFK_A1_WARP_MIN_HIDDEN
#define TFK_A1_WARP_MIN_HIDDEN 256
#endif
#ifndef TFK_A1_WARP_MAX_HIDDEN
#define TFK_A1_WARP_MAX_HIDDEN 6144
#endif

bool use_warp_kernel(int hidden) {
    int v = 0, threads = 0;
    if (hidden < 256 || hidden > 6144 || hidden < TFK_A1_WARP_MIN_HIDDEN || hidden > TFK_A1_WARP_MAX_HIDDEN ||
        !choose_shape(hidden, &v, &threads))
        return false;
    const bool exact = 8 * v * threads == hidden;
    return v == 3 || (v == 4 && !exact);
}

// Rows are handed out (when a workspace is given) only if each SM's share of
// x is at least this many bytes; below it every warp has only a few rows, the
// claims cost more than the balance brings, and the rows are split up front.
// Measured (fraction of the copy bandwidth, back to back, static / handed
// out): hidden 3072 at 4,000 rows 0.57 / 0.52, 8,192 0.71 / 0.68, 11,000
// 0.76 / 0.77, 14,600 0.79 / 0.82; hidden 1536 at 14,600 rows 0.74 / 0.70,
// 19,456 0.77 / 0.76, 29,000 0.80 / 0.82; hidden 6144 at 4,300 rows 0.64 /
// 0.66.  The crossing sits near 400 KB per SM for 1536 and 3072 and lower
// for 6144.
constexpr int64_t kHandOutMinBytesPerSm = 336 * 1024;

template <int VPL, bool kExact>
cudaError_t launch_warp(const AdalnArgs& a_in, int n_mod, cudaStream_t stream) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    AdalnArgs a = a_in;
    if (a.rows * a.hidden * 2 < kHandOutMinBytesPerSm * di.sm_count) a.sched = nullptr;
    const int64_t slot_bytes = (int64_t)a.hidden * 8;
    int64_t slots = ((int64_t)di.max_smem_per_block_optin - 2048) / slot_bytes;
    if (slots > n_mod) slots = n_mod;
    if (slots > kWarpMaxSlots) slots = kWarpMaxSlots;
    if (slots < 1) slots = 1;
    const size_t smem = (size_t)(slots * slot_bytes);
    const int64_t work = a.rows > a.padded_rows - a.rows ? a.rows : a.padded_rows - a.rows;
    // Few rows: smaller CTAs, so that the rows spread over all SMs.
    int64_t warps = (work + di.sm_count - 1) / di.sm_count;
    if (warps > kWarpThreads<VPL> / 32) warps = kWarpThreads<VPL> / 32;
    if (warps < 1) warps = 1;
    const int threads = (int)warps * 32;
    const void* fn = reinterpret_cast<const void*>(&rmsnorm_adaln_warp_kernel<VPL, kExact>);
    const int per_sm = blocks_per_sm(fn, threads, smem);
    if (per_sm <= 0) return cudaErrorInvalidConfiguration;
    int64_t grid = (work + warps - 1) / warps;
    if (grid > (int64_t)per_sm * di.sm_count) grid = (int64_t)per_sm * di.sm_count;
    if (grid < 1) return cudaSuccess;
    return launch_kernel(rmsnorm_adaln_warp_kernel<VPL, kExact>, (unsigned)grid, threads, smem, stream, a,
                         (int)slots, n_mod);
}

// Vectors per lane: the rows use_warp_kernel() admits have 192-640 vectors,
// i.e. 6, 9, 12, 15 or 17-20 per lane.
cudaError_t launch_warp_shape(const AdalnArgs& a, int n_mod, cudaStream_t stream) {
    const int nvec = a.hidden / 8;
    const int vpl = (nvec + 31) / 32;
    const bool whole = nvec % 32 == 0;
    if (vpl <= 6) return whole && vpl == 6 ? launch_warp<6, true>(a, n_mod, stream) : launch_warp<6, false>(a, n_mod, stream);
    if (vpl <= 12)
        return whole && vpl == 12 ? launch_warp<12, true>(a, n_mod, stream) : launch_warp<12, false>(a, n_mod, stream);
    if (vpl <= 16) return launch_warp<16, false>(a, n_mod, stream);
    if (vpl <= 20) return launch_warp<20, false>(a, n_mod, stream);
    return whole && vpl == 24 ? launch_warp<24, true>(a, n_mod, stream) : launch_warp<24, false>(a, n_mod, stream);
}

// Rows of more than 2176 vectors (hidden 17416 and wider): a pair of CTAs per
// row, each with the four-vector shape on its half (at most 2048 vectors, 512
// threads).  Measured against eight vectors per thread in one CTA, which spill
// (fraction of the copy bandwidth, 10,000 rows, event-timed): 18432 0.33 ->
// 0.39, 20480 0.35 -> 0.42, 24576 0.40 -> 0.45, 32768 0.46 -> 0.49; at 16392
// and 17408 the single CTA stays ahead (0.30 vs 0.28, 0.32 vs 0.30).  What
// holds the pairs back is the per-row cluster barrier: its release waits for
// the arriving threads' earlier memory operations, and the same kernel with
// a relaxed arrive (which does not make the exchanged sums visible, so a
// measurement only) ran at 0.63 at 20480 and 0.72 at 32768.
#ifndef TFK_A1_PAIR_FROM_NVEC
#define TFK_A1_PAIR_FROM_NVEC 2176
#endif
template <bool kExact>
cudaError_t launch_pair(const AdalnArgs& a, int threads, cudaStream_t stream) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    const int half = (a.hidden / 8 + 1) / 2;
    const int row_bytes = half * 16;
    auto kern = rmsnorm_adaln_kernel<4, kMaxThreads, kExact, true>;
    const void* fn = reinterpret_cast<const void*>(kern);
    const int by_regs = blocks_per_sm(fn, threads, 0);
    if (by_regs <= 0) return cudaErrorInvalidConfiguration;
    const int stages = pick_stages(by_regs, row_bytes, 0, row_bytes >= 16384 ? 80 * 1024 : kInflightPerSm);
    const size_t smem = (size_t)stages * row_bytes;
    const int per_sm = blocks_per_sm(fn, threads, smem);
    if (per_sm <= 0) return cudaErrorInvalidConfiguration;
    int64_t pairs = (int64_t)per_sm * di.sm_count / 2;
    if (pairs < 1) pairs = 1;
    const int64_t work = a.rows > a.padded_rows - a.rows ? a.rows : a.padded_rows - a.rows;
    const int64_t chunks = (work + kRowsPerCtaWide - 1) / kRowsPerCtaWide;
    if (chunks > pairs && work >= kChunkMinRun * pairs) pairs = chunks;
    if (pairs > (1 << 23)) pairs = 1 << 23;
    if (pairs > work) pairs = work;
    if (pairs < 1) return cudaSuccess;
    return launch_kernel_cluster(kern, (unsigned)(2 * pairs), threads, smem, 2, stream, a, stages);
}

}  // namespace

bool rmsnorm_adaln_supported(int hidden) {
    int v, t;
    return hidden > 0 && hidden % 8 == 0 && choose_shape(hidden, &v, &t);
}

cudaError_t launch_rmsnorm_adaln(const AdalnArgs& a, int n_mod, cudaStream_t stream) {
    if (use_warp_kernel(a.hidden)) return launch_warp_shape(a, n_mod, stream);
    const int nvec = a.hidden / 8;
    if (nvec > TFK_A1_PAIR_FROM_NVEC) {
        const int half = (nvec + 1) / 2;
        const int threads = ((half + 3) / 4 + 31) / 32 * 32;
        const bool exact = nvec % 2 == 0 && 4 * threads == half;
        return exact ? launch_pair<true>(a, threads, stream) : launch_pair<false>(a, threads, stream);
    }
    int v = 0, threads = 0;
    if (!choose_shape(a.hidden, &v, &threads)) return cudaErrorInvalidValue;
    const bool exact = 8 * v * threads == a.hidden;
    switch (v) {
        case 1: return launch_v<1, kMaxThreadsV1, false>(a, threads, stream);
        case 2:
            if (threads <= 256)
                return exact ? launch_v<2, 256, true>(a, threads, stream) : launch_v<2, 256, false>(a, threads, stream);
            return launch_v<2, kMaxThreads, false>(a, threads, stream);
        case 3: return launch_v<3, 256, true>(a, threads, stream);
        case 4:
            return exact ? launch_v<4, kMaxThreads, true>(a, threads, stream)
                         : launch_v<4, kMaxThreads, false>(a, threads, stream);
        default: return launch_v<8, kMaxThreads, false>(a, threads, stream);
    }
}

}  // namespace tfk
