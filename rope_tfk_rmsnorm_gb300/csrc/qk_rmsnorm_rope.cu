// qk_rmsnorm_rope.cu - Q/K per-head RMSNorm fused with NeoX rotate-half RoPE.
//
// For q (weight wq) and k (weight wk), each token t and head h (D = head_dim):
//   n[d]       = v[d] * rsqrt(mean_d v^2 + eps) * w[d]
//   a_i        = pos[t] * theta^(-2i/D),  i < D/2
//   out[i]     = n[i] cos a_i - n[i+D/2] sin a_i
//   out[i+D/2] = n[i+D/2] cos a_i + n[i] sin a_i
// (TeleFuser PR #38, section 2: Q/K RMSNorm and RoPE fused, together with the
// Ulysses packing; TeleFuser PR #23, section Changes Made: the Q/K
// normalization with NeoX RoPE kernel.)
//
// Design (HBM-bound: 4 bytes per q/k element read + written, plus 4 B/token):
// - A head is served by G lanes (G = D/16 rounded up to a power of two);
//   lane l holds the 8-element vector l of the first half and vector l of the
//   second half, so every rotate-half pair sits in one thread and needs no
//   shuffle; the per-head sum of squares is a G-lane shuffle reduction.
// - A group of G lanes owns HPT heads of the same tensor (q or k), so its
//   weights stay in registers, and the 8 cos/sin values a lane needs for a
//   token are computed once, folded with the weights, and used for HPT heads;
//   the per-head 1/rms, a scalar, is applied after the rotation.  Nothing is shared across
//   warps: there is no barrier anywhere in the token loop.
// - The grid is 2-D: contiguous token runs x chunks of head groups (any head
//   count fits), persistent over the token runs.  Each thread streams its own
//   head vectors through a shared-memory ring with cp.async, stages-1 tokens
//   ahead, and reads back only the slots it copied itself.
// - Angles are reduced exactly in integer arithmetic: theta^(-2i/D)/(2 pi) is
//   held as a 64-bit fixed-point fraction of a turn F_i (computed once per
//   launch in fp64 on the host side and passed by value), pos * F_i mod 2^64
//   is the angle's fraction of a turn, and
//   its top 32 bits give an fp32 angle in [-pi, pi).  On that range the
//   hardware sin/cos approximations are accurate to about 4e-7 absolute, so
//   no fp64 and no range reduction is needed per token.
// - The output can go straight into the Ulysses all-to-all send layout
//   [groups][rows][heads/groups][D] (the Ulysses packing fused into this step,
//   TeleFuser PR #38, section 2): only the store address changes.
#include <cmath>

#include "common.cuh"
#include "kernels.h"

namespace tfk {
namespace {

// 160 threads = 20 lane groups of 8 (head_dim 128): all 80 q/k heads of a
// 40-head token in one CTA at 4 heads per group, at most 136 registers (three
// CTAs per SM at least).  CTAs take 4-token chunks and the hardware block
// scheduler balances the chunks over the SMs: measured on the GB300 at 75,600
// tokens this reaches ~103% of the measured HBM peak, against 88% for one
// persistent run of ~166 tokens per CTA (whose static split leaves some SMs
// idle at the end) and 85% with a 102-register cap; 4-token chunks measured
// 1-4% above 8 on all four workload shapes, 8 above 16 and 24.
// Four heads per lane group, every group full and no token streams (the
// head counts of every workload here: 24, 32, 40) take 2-token chunks and a
// 96-register cap (four CTAs per SM) instead: measured (fraction of the
// copy bandwidth, event-timed, against 4-token chunks and 136 registers)
// 8,192 x 24 heads 0.766 -> 0.788, 30,358 x 24 0.949 -> 0.960, 75,600 x 40
// 1.023 -> 1.029, 56,320 x 32 1.004 -> 1.011; 1-token chunks 0.69-0.89, 3
// tokens between the two.  With masked groups (25 heads: 0.87 -> 0.80) or
// token streams (6 heads: 0.73 -> 0.69) the same change loses, so those keep
// 4-token chunks and 136 registers.
constexpr int kMaxThreads = 160;
template <int HPT, bool kMasked, bool kStreams>
constexpr bool kDense = HPT == 4 && !kMasked && !kStreams;
template <int HPT, bool kMasked, bool kStreams>
constexpr int kMinBlocks = kDense<HPT, kMasked, kStreams> ? 4 : 3;
template <int HPT, bool kMasked, bool kStreams>
constexpr int64_t kRowsPerCta = kDense<HPT, kMasked, kStreams> ? 2 : 4;

__device__ __forceinline__ void rope_cos_sin(int32_t pos, uint64_t turn_fraction, float& c, float& s) {
    const uint64_t a = (uint64_t)(int64_t)pos * turn_fraction;        // mod 2^64 = mod one turn
    const int32_t top = (int32_t)(uint32_t)(a >> 32);                   // [-2^31, 2^31) -> [-pi, pi)
    const float angle = (float)top * 1.46291807926715968e-9f;           // 2 pi / 2^32
    __sincosf(angle, &s, &c);
}

// Fixed-point turn fractions of the D/2 RoPE frequencies of one launch,
// frac(theta^(-2i/D) / (2 pi)) * 2^64, in the lane-interleaved layout read by
// the kernel (frequency i = 8*l + e of lane l at ((e/2)*L + l)*2 + e%2).  They
// depend only on (theta, head_dim), so they are computed once per launch, in
// double precision, and passed by value.
struct RopeTable {
    unsigned long long f[256];
};

RopeTable make_rope_table(double theta, int head_dim) {
    RopeTable t;
    const int half = head_dim / 2, L = head_dim / 16;
    for (int i = 0; i < half; ++i) {
        const double f = std::pow(theta, -2.0 * (double)i / (double)head_dim);
        double turns = f * 0.15915494309189533577;  // 1 / (2 pi)
        turns -= std::floor(turns);
        double scaled = std::ldexp(turns, 64);
        if (scaled >= 18446744073709551615.0) scaled = 18446744073709549568.0;  // largest double below 2^64
        const int l = i >> 3, e = i & 7;
        t.f[((e >> 1) * L + l) * 2 + (e & 1)] = (unsigned long long)scaled;
    }
    return t;
}

struct Layout {
    int hpt;          // heads per lane group (all of one tensor)
    int lanes;        // G
    int threads;      // per CTA
    int groups;       // lane groups in the whole problem: 2 * ceil(n_heads / hpt)
    int head_chunks;  // CTAs along the head dimension
    int groups_per_cta;  // lane groups of one token stream of a CTA
    int streams;      // token streams per CTA (side by side, each its own rows)
};

template <int HPT, bool kMasked, bool kStreams>
__global__ void __launch_bounds__(kMaxThreads, (kMinBlocks<HPT, kMasked, kStreams>)) qk_rope_kernel(const QkRopeArgs a, const Layout lay,
                                                              const int token_chunks, const int stages,
                                                              const __grid_constant__ RopeTable tab) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int nt = blockDim.x;
    const int tid = threadIdx.x;
    const int D = a.head_dim;
    const int half = D >> 1;
    const int L = D >> 4;                 // lanes holding data per head
    const int G = lay.lanes;
    const float inv_d = 1.0f / (float)D;

    Vec8* ring = reinterpret_cast<Vec8*>(smem_raw);                   // [stages][HPT][2][nt]
    const int stage_vecs = HPT * 2 * nt;
    uint64_t* ftab = reinterpret_cast<uint64_t*>(ring + (int64_t)stages * stage_vecs);  // [half]

    const int tchunk = blockIdx.x % token_chunks;
    const int hchunk = blockIdx.x / token_chunks;
    // A CTA may run several token streams side by side (to fill its warps when
    // one stream's lane groups leave lanes idle); stream s takes part s of the
    // CTA's token run.  Nothing below synchronises across groups: the only
    // barrier is the table copy above, and each head's reduction is a shuffle
    // within its own aligned G-lane group.
    const int gi = tid / G;
    const int nstreams = kStreams ? lay.streams : 1;
    int sidx = 0;
    if constexpr (kStreams) sidx = gi / lay.groups_per_cta < nstreams ? gi / lay.groups_per_cta : nstreams - 1;
    const int64_t c0 = a.rows * (int64_t)tchunk / token_chunks;
    const int64_t c1 = a.rows * (int64_t)(tchunk + 1) / token_chunks;
    const int64_t r0 = kStreams ? c0 + (c1 - c0) * sidx / nstreams : c0;
    const int nrows = (int)((kStreams ? c0 + (c1 - c0) * (sidx + 1) / nstreams : c1) - r0);

    // The launch's frequency table into shared memory (lane-interleaved layout:
    // the lanes of a warp then read consecutive 16-byte pairs, no bank conflicts).
    for (int i = tid; i < half; i += nt) ftab[i] = tab.f[i];
    __syncthreads();
    grid_dep_wait();

    const int lane = tid % G;
    const int group = hchunk * lay.groups_per_cta + (gi - sidx * lay.groups_per_cta);
    const bool active = gi < nstreams * lay.groups_per_cta && group < lay.groups && lane < L;
    // Groups 0 .. gq-1 take the q heads HPT at a time, the next gq the k heads;
    // the last group of each tensor may hold fewer than HPT heads (nvalid).
    const int gq = (a.n_heads + HPT - 1) / HPT;
    const bool is_q = group < gq;
    const int h0 = (is_q ? group : group - gq) * HPT;
    const int nvalid = !kMasked ? HPT : (a.n_heads - h0 < HPT ? a.n_heads - h0 : HPT);
    const uint16_t* src0 = (is_q ? a.q : a.k) + (int64_t)h0 * D + lane * 8;
    uint16_t* outp = is_q ? a.q_out : a.k_out;
    const float* wsrc = is_q ? a.q_weight : a.k_weight;
    f32x2 wa[4], wb[4];  // weights of this lane's first-half / second-half elements, as pairs
    const ulonglong2* fq = reinterpret_cast<const ulonglong2*>(ftab) + (active ? lane : 0);  // stride L per pair
    if (active) {
        const float4 x0 = ld_f4(wsrc + lane * 8), x1 = ld_f4(wsrc + lane * 8 + 4);
        const float4 y0 = ld_f4(wsrc + half + lane * 8), y1 = ld_f4(wsrc + half + lane * 8 + 4);
        wa[0] = f2_make(x0.x, x0.y); wa[1] = f2_make(x0.z, x0.w); wa[2] = f2_make(x1.x, x1.y); wa[3] = f2_make(x1.z, x1.w);
        wb[0] = f2_make(y0.x, y0.y); wb[1] = f2_make(y0.z, y0.w); wb[2] = f2_make(y1.x, y1.y); wb[3] = f2_make(y1.z, y1.w);
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) { wa[k] = 0ull; wb[k] = 0ull; }
    }
    // Output offset of each of the group's heads (token 0): output group
    // h / hpg at group_stride, head h % hpg inside that group's row (in the
    // Ulysses layout consecutive heads may fall in different groups).
    int64_t out_off[HPT];
#pragma unroll
    for (int j = 0; j < HPT; ++j) {
        const int h = h0 + j;
        const int ogrp = h / a.heads_per_group;
        out_off[j] = (int64_t)ogrp * a.group_stride + (int64_t)(h - ogrp * a.heads_per_group) * D + lane * 8;
    }

    auto issue = [&](int row_in_run, int stage) {
        const uint16_t* src = src0 + (r0 + row_in_run) * a.in_stride;
        Vec8* st = ring + (int64_t)stage * stage_vecs + tid;
#pragma unroll
        for (int j = 0; j < HPT; ++j) {
            if (j < nvalid) {
                cp_async16(st + (j * 2 + 0) * nt, src + j * D);
                cp_async16(st + (j * 2 + 1) * nt, src + j * D + half);
            }
        }
    };

    // nrows is uniform over one token stream, not over the CTA: with kStreams
    // the streams of a CTA leave this loop at different iterations.  That is
    // safe only because the loop holds no CTA-wide barrier and no full-warp
    // collective: every shuffle below uses the mask of its own G-lane group,
    // which never spans two streams (a stream owns whole groups).  Adding a
    // __syncthreads or a full-warp reduction inside this loop would deadlock
    // whenever kStreams is set.
    if (nrows > 0) {
        for (int s = 0; s < stages - 1; ++s) {
            if (active && s < nrows) issue(s, s);
            cp_async_commit();
        }
        int stage_rd = 0, stage_wr = stages - 1;
        int32_t p_next = __ldg(a.pos + r0);
        for (int it = 0; it < nrows; ++it) {
            const int64_t r = r0 + it;
            const int ahead = it + stages - 1;
            if (active && ahead < nrows) issue(ahead, stage_wr);
            cp_async_commit();
            stage_wr = stage_wr + 1 == stages ? 0 : stage_wr + 1;
            const int32_t p = p_next;
            if (it + 1 < nrows) p_next = __ldg(a.pos + r + 1);

            // Weights folded into the rotation once per token for all HPT heads:
            //   out[i]     = inv_rms * (v[i] * wa*c - v[i+D/2] * wb*s)
            //   out[i+D/2] = inv_rms * (v[i+D/2] * wb*c + v[i] * wa*s)
            // (the per-head 1/rms is a scalar, so it can be applied after the rotation).
            f32x2 wac[4], nwbs[4], wbc[4], was[4];  // wa*c, -(wb*s), wb*c, wa*s per element pair
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const ulonglong2 fpair = fq[k * L];
                float c0, s0, c1, s1;
                rope_cos_sin(p, fpair.x, c0, s0);
                rope_cos_sin(p, fpair.y, c1, s1);
                const f32x2 c2 = f2_make(c0, c1), s2 = f2_make(s0, s1), ns2 = f2_make(-s0, -s1);
                wac[k] = f2_mul(wa[k], c2);
                nwbs[k] = f2_mul(wb[k], ns2);
                wbc[k] = f2_mul(wb[k], c2);
                was[k] = f2_mul(wa[k], s2);
            }

            cp_async_wait_dyn(stages - 1);
            const Vec8* st = ring + (int64_t)stage_rd * stage_vecs + tid;
            stage_rd = stage_rd + 1 == stages ? 0 : stage_rd + 1;

            float ss[HPT];
#pragma unroll
            for (int j = 0; j < HPT; ++j) {
                const Vec8 a8 = ld_smem_vec(st + (j * 2 + 0) * nt), b8 = ld_smem_vec(st + (j * 2 + 1) * nt);
                f32x2 sa = 0ull, sb = 0ull;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const f32x2 va = bf2_to_f2(a8.w[k]), vb = bf2_to_f2(b8.w[k]);
                    sa = f2_fma(va, va, sa);
                    sb = f2_fma(vb, vb, sb);
                }
                float a0, a1, b0, b1;
                f2_split(sa, a0, a1);
                f2_split(sb, b0, b1);
                ss[j] = active && j < nvalid ? (a0 + a1) + (b0 + b1) : 0.f;
            }
            for (int o = G >> 1; o > 0; o >>= 1) {
#pragma unroll
                for (int j = 0; j < HPT; ++j) {
                    if constexpr (kStreams) {  // lanes of other streams may have left the loop
                        const unsigned gmask = G == 32 ? 0xFFFFFFFFu : ((1u << G) - 1u) << ((tid & 31) & ~(G - 1));
                        ss[j] += __shfl_xor_sync(gmask, ss[j], o);
                    } else {
                        ss[j] += __shfl_xor_sync(0xFFFFFFFFu, ss[j], o);
                    }
                }
            }
            if (active) {
                const int64_t roff = r * a.out_stride;
#pragma unroll
                for (int j = 0; j < HPT; ++j) {
                    if (j >= nvalid) continue;
                    const Vec8 a8 = ld_smem_vec(st + (j * 2 + 0) * nt), b8 = ld_smem_vec(st + (j * 2 + 1) * nt);
                    const float inv_rms = rsqrtf(ss[j] * inv_d + a.eps);
                    const f32x2 inv2 = f2_make(inv_rms, inv_rms);
                    Vec8 oa, ob;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const f32x2 va = bf2_to_f2(a8.w[k]), vb = bf2_to_f2(b8.w[k]);
                        oa.w[k] = f2_to_bf2(f2_mul(f2_fma(va, wac[k], f2_mul(vb, nwbs[k])), inv2));
                        ob.w[k] = f2_to_bf2(f2_mul(f2_fma(vb, wbc[k], f2_mul(va, was[k])), inv2));
                    }
                    uint16_t* o = outp + out_off[j] + roff;
                    st_vec(o, oa);
                    st_vec(o + half, ob);
                }
            }
        }
        cp_async_wait<0>();
    }  // nrows > 0

    // Fixed-valid mode: this CTA's share of the padded tail rows of q_out and
    // k_out is written +0.0 in the same launch (the input tail is never read).
    const int64_t tail = a.padded_rows - a.rows;
    if (tail > 0 && active) {
        const int64_t t0 = a.rows + tail * (int64_t)tchunk / token_chunks;
        const int64_t t1 = a.rows + tail * (int64_t)(tchunk + 1) / token_chunks;
        const int64_t z0 = t0 + (t1 - t0) * sidx / nstreams;
        const int64_t z1 = t0 + (t1 - t0) * (sidx + 1) / nstreams;
        Vec8 zero;
        zero.w[0] = zero.w[1] = zero.w[2] = zero.w[3] = 0u;
        for (int64_t r = z0; r < z1; ++r) {
            const int64_t roff = r * a.out_stride;
#pragma unroll
            for (int j = 0; j < HPT; ++j) {
                if (j >= nvalid) continue;
                uint16_t* o = outp + out_off[j] + roff;
                st_vec(o, zero);
                st_vec(o + half, zero);
            }
        }
    }
}

// heads_per_group: heads per output group (n_heads, or n_heads / sp_degree in
// the Ulysses layout).  A lane group's heads are all q or all k; they may
// fall in different output groups.  Four heads per group from 4 heads on, the
// last group of each tensor masked when 4 does not divide n_heads: the
// per-token cos/sin work is then shared by up to 4 heads even for odd head
// counts (25 x 128: 55% -> 94% of the copy bandwidth; 30 x 96: 66% -> 86%).
bool choose_layout(int n_heads, int head_dim, int heads_per_group, Layout* lay) {
    if (head_dim < 16 || head_dim > 512 || head_dim % 16 != 0 || n_heads < 1 || n_heads > (1 << 20)) return false;
    if (heads_per_group < 1 || n_heads % heads_per_group != 0) return false;
    int L = head_dim / 16, G = 1;
    while (G < L) G <<= 1;
    // 3 heads per group for 3, 6 and 9 heads, where groups of 4 would leave a
    // quarter of their head slots masked (6 x 128: 88% -> 94%); elsewhere 4
    // heads per group measured ahead even with idle lanes or masked heads
    // (25 x 128: 95% with 4 against 86% with 3; 12 x 128 within 1%).
    int hpt = n_heads >= 4 ? 4 : (n_heads >= 2 ? 2 : 1);
    if (n_heads % 3 == 0 && n_heads % 4 != 0 && n_heads <= 9) hpt = 3;
    const int64_t groups = 2LL * ((n_heads + hpt - 1) / hpt);
    // as few head chunks as possible with at most kMaxThreads threads per CTA
    const int64_t per_cta = kMaxThreads / G;
    const int64_t chunks = (groups + per_cta - 1) / per_cta;
    const int64_t groups_per_cta = (groups + chunks - 1) / chunks;
    // Few heads (all lane groups of a token in at most half a warp): token
    // streams side by side fill the warp (3 x 128: 59% -> 80% of the copy
    // bandwidth).  Measured and left out for wider layouts whose last warp is
    // only partly idle (12 x 128: 90% -> 85%, 20 x 128: 97% -> 88%).
    int streams = 1;
    const int64_t lanes = groups_per_cta * G;
    if (chunks == 1 && lanes <= 16) streams = (int)(32 / lanes);
    const int64_t threads = (streams * lanes + 31) / 32 * 32;
    lay->groups_per_cta = (int)groups_per_cta;
    lay->streams = streams;
    lay->hpt = hpt;
    lay->lanes = G;
    lay->threads = (int)threads;
    lay->groups = (int)groups;
    lay->head_chunks = (int)chunks;
    return chunks <= 65535;
}

template <int HPT, bool kMasked, bool kStreams>
cudaError_t launch_h(const QkRopeArgs& a, const Layout& lay, cudaStream_t stream) {
    DeviceInfo di;
    cudaError_t err = device_info(&di);
    if (err != cudaSuccess) return err;
    const int stage_bytes = HPT * 2 * lay.threads * 16;
    const int table_bytes = (a.head_dim / 2) * 8;
    const void* fn = reinterpret_cast<const void*>(&qk_rope_kernel<HPT, kMasked, kStreams>);
    const int by_regs = blocks_per_sm(fn, lay.threads, table_bytes + 2 * stage_bytes);
    if (by_regs <= 0) return cudaErrorInvalidConfiguration;
    const int stages = pick_stages(by_regs, stage_bytes, table_bytes);
    const size_t smem = (size_t)stages * stage_bytes + table_bytes;
    const int per_sm = blocks_per_sm(fn, lay.threads, smem);
    if (per_sm <= 0) return cudaErrorInvalidConfiguration;
    // token runs: enough CTAs for every SM, and no more runs than rows to work on
    int64_t want = ((int64_t)per_sm * di.sm_count + lay.head_chunks - 1) / lay.head_chunks;
    const int64_t work = a.rows > a.padded_rows - a.rows ? a.rows : a.padded_rows - a.rows;
    {  // fixed-size chunks instead of one persistent run per CTA
        const int64_t per = kRowsPerCta<HPT, kMasked, kStreams> * lay.streams;  // rows per stream stay the chunk
        const int64_t chunks = (work + per - 1) / per;
        if (chunks > want) want = chunks;
    }
    if (want > (1 << 24)) want = 1 << 24;  // the token split covers any count; keeps rows * chunk in range
    if (want > work) want = work;
    if (want < 1) return cudaSuccess;
    const int64_t grid = want * lay.head_chunks;
    if (grid > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    // the table of the last (theta, head_dim) seen on this host thread is kept
    thread_local float last_theta = -1.0f;
    thread_local int last_dim = 0;
    thread_local RopeTable table;
    if (a.theta != last_theta || a.head_dim != last_dim) {
        table = make_rope_table(a.theta, a.head_dim);
        last_theta = a.theta;
        last_dim = a.head_dim;
    }
    return launch_kernel(qk_rope_kernel<HPT, kMasked, kStreams>, (unsigned)grid, lay.threads, smem, stream, a, lay, (int)want, stages,
                         table);
}

}  // namespace

bool qk_rope_supported(int n_heads, int head_dim) {
    Layout lay;
    return choose_layout(n_heads, head_dim, n_heads, &lay);
}

cudaError_t launch_qk_rmsnorm_rope(const QkRopeArgs& a, cudaStream_t stream) {
    Layout lay;
    if (!choose_layout(a.n_heads, a.head_dim, a.heads_per_group, &lay)) return cudaErrorInvalidValue;
    const bool masked = a.n_heads % lay.hpt != 0;  // separate instantiations: no predicates otherwise
    const bool streams = lay.streams > 1;
#define TFK_QK_LAUNCH(H) \
    (masked ? (streams ? launch_h<H, true, true>(a, lay, stream) : launch_h<H, true, false>(a, lay, stream)) \
            : (streams ? launch_h<H, false, true>(a, lay, stream) : launch_h<H, false, false>(a, lay, stream)))
    switch (lay.hpt) {
        case 1: return streams ? launch_h<1, false, true>(a, lay, stream) : launch_h<1, false, false>(a, lay, stream);
        case 2: return TFK_QK_LAUNCH(2);
        case 3: return TFK_QK_LAUNCH(3);
        default: return TFK_QK_LAUNCH(4);
    }
#undef TFK_QK_LAUNCH
}

}  // namespace tfk
