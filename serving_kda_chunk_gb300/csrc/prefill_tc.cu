// prefill_tc.cu -- chunked KDA prefill on the Blackwell tensor cores.
//
// One CTA per (sequence, head) walks the sequence in chunks of C = 64 tokens
// with the fp32 state held in tensor memory (TMEM) for the whole sequence;
// every dense contraction of a chunk runs on tcgen05 with fp32 accumulation.
//
// Chunk form of the recurrence (the WY / UT-transform products, Q K^T, K S and
// K^T U tiles; G_t = sum_{u<=t} g_u inside the chunk, per key channel):
//   A_ts = sum_i k_ti k_si e^{G_ti - G_si} (s < t),  P_ts = sum_i q_ti k_si e^{G_ti - G_si} (s <= t)
//   T    = (I + Diag(beta) A)^-1,        T_b = T Diag(beta)
//   W    = T_b (k e^{G}),                U~  = T_b V
//   U    = U~ - W S,                     O   = (q e^{G}) S + P U
//   S   <- Diag(e^{G_63}) S + (k e^{G_63 - G})^T U
// Everything is computed transposed so that the 128-wide value / key axis is
// the MMA M dimension (M = 128 for every product):
//   [A;P]  = [L_k; L_q] R^T          (M = 2x64 stacked rows, N = 64, K = 128)
//   W^T    = (k e^G)^T T_b^T,  U~^T = V^T T_b^T      (M = 128, N = 64, K = 64)
//   U^T    = U~^T - S^T W^T,   O^T = S^T (q e^G)^T    (M = 128, N = 64, K = 128)
//   O^T   += U^T P^T,          S^T <- S^T Diag(e^{G_63}) + U^T (k e^{G_63-G})  (K = 64)
// with L = k e^{G_t - G_31}, R = k e^{G_31 - G_s} (reference at the chunk
// middle, so each factor spans at most 32 tokens).  The intra-chunk decays are
// formed as running products of alpha = 1/(1+e^x) and 1/alpha = 1+e^x, so a
// chunk costs two transcendental evaluations per (token, channel).
//
// Precision: operands that are not exact bf16 inputs are split into bf16
// hi + lo and their products formed as hi*hi + hi*lo + lo*hi (relative error
// ~2^-17); with bf16 outputs the two products that only feed the output
// (S^T Q^T, U^T P^T) use hi only.  The state stays fp32 in TMEM.  If a half
// chunk's cumulative decay leaves the range those factors can carry (a factor
// above 2^64), that chunk is evaluated token by token on CUDA cores instead.
//
// Work split: 512 threads.  TMEM passes: warp w reads lanes 32*(w%4)..+31 and
// the column quarter w/4 of a tile.  Channel passes (gates, decayed operands):
// thread (key channel tid%128, token quarter tid/128), 16 tokens each; the
// running decay products start from the other quarters' totals, exchanged
// through shared memory.
//
// The snapshot of chunk j (the state after j*64 tokens of the sequence, SGLang
// PR 34820 page, the fp32 track-state snapshot) is written from the fp32 TMEM
// accumulator when chunk j starts; with a 16-bit state type it is that
// accumulator rounded once, like the initial / final states of the pool.
#include "kda_common.cuh"
#include "kda_host.h"
#include "prefill.h"
#include "umma.cuh"

namespace kda {
namespace {

using namespace umma;

constexpr int kThreads = 512;  // 16 warps: four per TMEM lane quarter
constexpr int kTrackTc = 512;  // snapshot requests per sequence handled by this kernel

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_RAW = 0;      // raw q, k, g tiles of the chunk, row-major bf16 [t][128]
constexpr uint32_t OFF_X = 49152;    // 96 KiB reused by the chunk phases:
//   fallback alpha (fp32 [64][128]), dot scratch     X+0, X+32K
//   L hi/lo (A, MN-major, M = 128, K = 128)          X+0,  X+32K
//   [R hi; R lo] (B, MN-major, N = 2 x 64, K = 128)  X+64K, X+80K
//   N^T, T (fp32 [64][68]) and solve temporaries     X+0 .. X+41K
//   [QG; -W hi; -W lo] (B, MN-major, N = 3 x 64)     X+0, X+16K, X+32K
//   [KT hi; P] (B, K-major, 128 + 64 rows), KT lo    X+48K, X+64K, X+72K
//   P lo (fp32 outputs)                              X+88K
constexpr uint32_t OFF_V = OFF_X + 98304;  // A: V, MN-major (c atoms 8 KiB apart, s groups 1 KiB),
                                           // two buffers (chunk parity) 16 KiB apart
constexpr uint32_t OFF_TB_HI = OFF_V + 32768;    // B: [T_b hi; T_b lo] [t][s], K-major, 64 + 64 rows
constexpr uint32_t OFF_TB_LO = OFF_TB_HI + 8192;
constexpr uint32_t OFF_QG_LO = OFF_TB_LO + 8192;  // QG lo (fp32 outputs), MN-major
constexpr uint32_t OFF_MISC = OFF_QG_LO + 16384;
constexpr uint32_t MISC_BYTES = 8192;
constexpr uint32_t SMEM_BYTES = OFF_MISC + MISC_BYTES + 1024;  // + alignment slack

constexpr uint32_t RAW_Q = OFF_RAW, RAW_K = OFF_RAW + 16384, RAW_G = OFF_RAW + 32768;
constexpr uint32_t X_ALPHA = OFF_X, X_RED = OFF_X + 32768;
constexpr uint32_t X_L_HI = OFF_X, X_L_LO = OFF_X + 32768, X_R_HI = OFF_X + 65536,
                   X_R_LO = OFF_X + 81920;
constexpr uint32_t X_N = OFF_X, X_T = OFF_X + 17408, X_Y1 = OFF_X + 34816, X_Y2 = OFF_X + 37376;
constexpr uint32_t X_QG = OFF_X, X_W_HI = OFF_X + 16384, X_W_LO = OFF_X + 32768;
constexpr uint32_t X_KT_HI = OFF_X + 49152, X_P = OFF_X + 65536, X_KT_LO = OFF_X + 73728,
                   X_P_LO = OFF_X + 90112;
constexpr int NLD = 68;  // fp32 row stride of the N / T matrices

// TMEM columns: fp32 accumulators, and bf16 hi/lo A operands (two per column) whose rows are
// the TMEM lanes.  A tcgen05.mma costs about the same for any N up to 256, so products that
// share an A operand are issued as one MMA over B tiles laid side by side, into adjacent
// accumulators: [S | O] takes U^T [KT; P], [O | U_a | U_b] takes S^T [QG; -W hi; -W lo].
constexpr uint32_t TM_S = 0;                     // S^T, fp32, 128 columns
constexpr uint32_t TM_O = 128;                   // O^T (W^T while MMA 2 runs)
constexpr uint32_t TM_UA = 192, TM_UB = 256;     // U^T = U_a + U_b (hi and lo T_b parts)
constexpr uint32_t TM_AP = 192;                  // [A; P] as hi + lo parts (MMA 1 only)
constexpr uint32_t TM_SA_HI = 320, TM_SA_LO = 384;  // S^T [c][i], K = 128
constexpr uint32_t TM_KG_HI = 448, TM_KG_LO = 480;  // KG [i][s], K = 64 (until MMA 2)
constexpr uint32_t TM_U_HI = 448, TM_U_LO = 480;    // U^T [c][s], K = 64 (from MMA 3 on)
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t kWaitLimit = 1u << 18;    // polls of ~4 us (try_wait suspends): ~1 s; a healthy MMA batch takes microseconds
constexpr float kFactorMax = 1.8446744e19f;  // 2^64

__device__ __forceinline__ float bf16_at(const uint8_t* sm, uint32_t off) {
    return __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t*>(sm + off)) << 16);
}

__device__ __forceinline__ void st16(uint8_t* sm, uint32_t off, uint4 v) {
    *reinterpret_cast<uint4*>(sm + off) = v;
}

template <bool kBf16Out>
__global__ void __launch_bounds__(kThreads, 1) prefill_tc_kernel(PrefillArgs p,
                                                                 const int32_t* __restrict__ order) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(sm);
    const uint32_t sb4 = sb >> 4;  // descriptor units
    float* s_beta = reinterpret_cast<float*>(sm + OFF_MISC);  // 64
    float* s_gam = s_beta + 64;                               // 128: e^{G_63}
    float* s_seg_a = s_gam + 128;                             // [4][128]: prod of alpha per token quarter
    float* s_seg_i = s_seg_a + 512;                           // [4][128]: prod of 1/alpha per quarter
    int* s_trk = reinterpret_cast<int*>(s_seg_i + 512);       // kTrackTc
    uint64_t* s_mbar = reinterpret_cast<uint64_t*>(s_trk + kTrackTc);  // [0]: MMA batches, [1]: state update
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(s_mbar + 2);
    int* s_abort = reinterpret_cast<int*>(s_tmem + 1);  // a wait that timed out inside a phase
    float* s_nk = reinterpret_cast<float*>(s_abort + 4);  // 64: L2 factors of the key rows
    float* s_nq = s_nk + 64;                              // 64: of the query rows (x scale)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool l2 = (p.flags & KDA_QK_L2NORM) != 0;
    // raw key / query element (t, ch) as the recurrence uses it (q also times scale; under
    // KDA_QK_L2NORM each row times its L2 factor)
    auto key_at = [&](int t, int ch) {
        const float x = bf16_at(sm, RAW_K + t * 256 + ch * 2);
        return l2 ? x * s_nk[t] : x;
    };
    auto query_at = [&](int t, int ch) {
        const float x = bf16_at(sm, RAW_Q + t * 256 + ch * 2);
        return l2 ? x * s_nq[t] : x * p.scale;
    };
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int cq = warp >> 2;      // column quarter this warp takes in TMEM passes
    const int row = quarter * 32 + lane;
    const int ci = tid & 127, tq = tid >> 7;  // channel passes: key channel, token quarter
    const int H = p.H;
    const int unit = blockIdx.x;
    const int n = order ? order[unit / H] : unit / H;
    const int h = unit - (unit / H) * H;

    const int t0 = p.cu_seqlens[n], t1 = p.cu_seqlens[n + 1];
    if (t0 < 0 || t1 < t0 || t1 > p.T_tot || (n == 0 && t0 != 0)) {
        if (tid == 0 && h == 0) report(p.dev_status, KDA_DEV_BAD_SEQLEN);
        return;
    }
    const int L = t1 - t0;
    const int n_chunks = (L + kChunk - 1) / kChunk;
    const int init = p.init_slot ? p.init_slot[n] : -1;
    const int fin = p.final_slot ? p.final_slot[n] : -1;
    if (init >= p.P || fin >= p.P) {
        if (tid == 0 && h == 0) report(p.dev_status, KDA_DEV_BAD_SLOT);
        return;
    }
    for (int m = tid; m < p.M; m += kThreads) {
        const int j = p.track[(size_t)n * p.M + m];
        const bool ok = j >= -1 && j < n_chunks;
        if (!ok && h == 0) report(p.dev_status, KDA_DEV_BAD_TRACK);
        s_trk[m] = ok ? j : -1;
    }

    // ---- TMEM and the MMA completion barriers
    if (warp == 0) tmem_alloc(smem_u32(s_tmem), TM_COLS);
    if (tid == 0) {
        mbar_init(smem_u32(s_mbar), 1);
        mbar_init(smem_u32(s_mbar + 1), 1);
        *s_abort = 0;
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);  // this warp's lanes
    const uint32_t mbar = smem_u32(s_mbar);      // MMA batches whose results threads read
    const uint32_t mbar_s = smem_u32(s_mbar + 1);  // the state update, waited one chunk later
    uint32_t phase = 0, phase_s = 0;
    bool pending_s = false;

    // ---- initial state into TMEM (row c = S^T row, this warp's 32 columns)
    {
        const size_t S0 = init >= 0 ? state_elem(init, H, h) + (size_t)row * kD : 0;
        const int col0 = cq * 32;
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            float4 x = init >= 0 ? state_load4(p.pool, S0 + col0 + j, p.st)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
            v[j] = x.x;
            v[j + 1] = x.y;
            v[j + 2] = x.z;
            v[j + 3] = x.w;
        }
        st32(tl + TM_S + col0, v);
        wait_st();
    }

    bool timed_out = false;
    const __nv_bfloat16* gq = static_cast<const __nv_bfloat16*>(p.q);
    const __nv_bfloat16* gk = static_cast<const __nv_bfloat16*>(p.k);
    const __nv_bfloat16* gv = static_cast<const __nv_bfloat16*>(p.v);
    const __nv_bfloat16* gg = static_cast<const __nv_bfloat16*>(p.gate_raw);

    // Raw tiles of chunk jj arrive by cp.async: q, k, g row-major (free once the
    // decayed operands of the previous chunk are written), v as the MN-major MMA
    // operand in the buffer of the chunk's parity (requested one chunk ahead).
    // Rows past the sequence are zero-filled.
    auto prefetch_qkg = [&](int jj) {
        const int cn = t0 + jj * kChunk, ln = min(kChunk, t1 - cn);
#pragma unroll
        for (int it = tid; it < 64 * 16; it += kThreads) {
            const int t = it >> 4, ch = it & 15;
            const bool ok = t < ln;
            const size_t e = ok ? ((size_t)(cn + t) * H + h) * kD + ch * 8 : 0;
            const uint32_t nb = ok ? 16u : 0u;
            cp_async16(sb + RAW_Q + t * 256 + ch * 16, gq + e, nb);
            cp_async16(sb + RAW_K + t * 256 + ch * 16, gk + e, nb);
            cp_async16(sb + RAW_G + t * 256 + ch * 16, gg + e, nb);
        }
    };
    auto prefetch_v = [&](int jj) {
        const int cn = t0 + jj * kChunk, ln = min(kChunk, t1 - cn);
        const uint32_t vb = OFF_V + (uint32_t)(jj & 1) * 16384;
#pragma unroll
        for (int it = tid; it < 64 * 16; it += kThreads) {
            const int t = it >> 4, ch = it & 15;
            const bool ok = t < ln;
            const size_t e = ok ? ((size_t)(cn + t) * H + h) * kD + ch * 8 : 0;
            cp_async16(sb + vb + chunk_mn(ch * 8, t, 8192, 1024), gv + e, ok ? 16u : 0u);
        }
    };
    // raw beta of chunk jj, loaded one chunk ahead and activated when the chunk starts; rows
    // past the sequence read its last token (never out of bounds) and get beta = 0 there.  No
    // select on the loaded value, so nothing waits for the load before its use.
    auto load_beta = [&](int jj) -> uint32_t {  // raw bf16 bits, widened when used
        const int cn = t0 + jj * kChunk, ln = min(kChunk, t1 - cn);
        return __ldg(static_cast<const unsigned short*>(p.beta_raw) + (size_t)(cn + min(tid, ln - 1)) * H + h);
    };
    uint32_t beta_next = 0;
    if (n_chunks > 0) {
        prefetch_qkg(0);
        prefetch_v(0);
        cp_async_commit();
        if (tid < 64) beta_next = load_beta(0);
    }

    for (int j = 0; j < n_chunks && !timed_out; ++j) {
        const int c0 = t0 + j * kChunk;
        const int Lc = min(kChunk, t1 - c0);
        const bool more = j + 1 < n_chunks;
        cp_async_wait_all();
        if (tid < 64) s_beta[tid] = tid < Lc ? beta_act(__uint_as_float(beta_next << 16), p.flags) : 0.f;
        fence_before();
        if (__syncthreads_or(timed_out)) {
            timed_out = true;
            break;
        }
        fence_after();
        if (tid < 64 && more) beta_next = load_beta(j + 1);  // lands during this chunk
        const uint32_t v_cur = OFF_V + (uint32_t)(j & 1) * 16384;
        if (more) {
            prefetch_v(j + 1);  // the other buffer's last reader was chunk j - 1
            cp_async_commit();
        }
        if (l2) {
            // KDA_QK_L2NORM: the factors of the key and query rows, a warp per 4 rows (first read
            // after the channel pass's barrier)
#pragma unroll
            for (int tt = 0; tt < 4; ++tt) {
                const int t = 4 * warp + tt;
                const float4 kx = State<kStateBF16>::widen(*reinterpret_cast<const uint2*>(sm + RAW_K + t * 256 + lane * 8));
                const float4 qx = State<kStateBF16>::widen(*reinterpret_cast<const uint2*>(sm + RAW_Q + t * 256 + lane * 8));
                float sk = f4_dot(kx, kx), sq = f4_dot(qx, qx);
                warp_sum2(sk, sq);
                if (lane == 0) {
                    s_nk[t] = l2norm_factor(sk);
                    s_nq[t] = l2norm_factor(sq) * p.scale;
                }
            }
        }

        // ---- channel pass: this thread's channel ci over tokens 16*tq .. 16*tq+15
        float al[16], iv[16];
        float m_big = 1.f;  // product of the factors >= 1 this quarter contributes to its half
        {
            with_gate_form(p.flags, [&](uint32_t form) {
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int t = 16 * tq + u;
                    const Decay dc = decay_of(bf16_at(sm, RAW_G + t * 256 + ci * 2), form);
                    al[u] = t < Lc ? dc.a : 1.f;
                    iv[u] = t < Lc ? dc.inv : 1.f;
                }
            });
            float pa = 1.f, pi = 1.f;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                pa *= al[u];
                pi *= iv[u];
                if (tq != 0 || u > 0) m_big *= iv[u];
            }
            s_seg_a[tq * 128 + ci] = pa;
            s_seg_i[tq * 128 + ci] = pi;
        }
        __syncthreads();
        bool bad = false;
        // largest factor a half uses: prod of 1/alpha over (0, 31] (half 0) or [32, 63] (half 1)
        if (tq == 0) bad = !(m_big * s_seg_i[128 + ci] <= kFactorMax);
        if (tq == 2) bad = !(m_big * s_seg_i[384 + ci] <= kFactorMax);
        // the previous chunk's state update (U^T, KT operands; S) must be complete before the
        // operand regions are rewritten and S is read: it ran behind this chunk's gate pass
        if (pending_s) {
            if (!mbar_wait(mbar_s, phase_s, kWaitLimit)) *s_abort = 1;
            phase_s ^= 1;
            pending_s = false;
        }
        fence_after();
        const int fallback = __syncthreads_or(bad);
        if (*s_abort) {
            timed_out = true;
            break;
        }

        if (!fallback) {
            // ---- L = [k; q] e^{G_t - G_31}, R = k e^{G_31 - G_s}: quarters 0, 1 backward
            //      from token 31, quarters 2, 3 forward from token 32
            if (tq < 2) {
                float sa = 1.f, si = 1.f;  // prod over (u, 31] of alpha and of 1/alpha
                if (tq == 0) {
                    sa = s_seg_a[128 + ci];
                    si = s_seg_i[128 + ci];
                }
#pragma unroll
                for (int g8 = 1; g8 >= 0; --g8) {
                    float lk[8], lq[8], r[8];
#pragma unroll
                    for (int w = 7; w >= 0; --w) {
                        const int u = g8 * 8 + w, t = 16 * tq + u;
                        const float kk = key_at(t, ci);
                        const float qq = query_at(t, ci);
                        lk[w] = kk * si;
                        lq[w] = qq * si;
                        r[w] = kk * sa;
                        sa *= al[u];
                        si *= iv[u];
                    }
                    uint4 hi, lo;
                    const int tt = 16 * tq + g8 * 8;
                    split8(lk, hi, lo);
                    st16(sm, X_L_HI + chunk_mn(tt, ci, 1024, 2048), hi);
                    st16(sm, X_L_LO + chunk_mn(tt, ci, 1024, 2048), lo);
                    split8(lq, hi, lo);
                    st16(sm, X_L_HI + chunk_mn(64 + tt, ci, 1024, 2048), hi);
                    st16(sm, X_L_LO + chunk_mn(64 + tt, ci, 1024, 2048), lo);
                    split8(r, hi, lo);
                    st16(sm, X_R_HI + chunk_mn(tt, ci, 1024, 1024), hi);
                    st16(sm, X_R_LO + chunk_mn(tt, ci, 1024, 1024), lo);
                }
                if (tq == 0) {
                    const float a0 = s_seg_a[ci], a1 = s_seg_a[128 + ci], a2 = s_seg_a[256 + ci],
                                a3 = s_seg_a[384 + ci];
                    s_gam[ci] = (a0 * a1) * (a2 * a3);  // e^{G_63}
                }
            } else {
                float fa = 1.f, fi = 1.f;  // prod over [32, t] of alpha and of 1/alpha
                if (tq == 3) {
                    fa = s_seg_a[256 + ci];
                    fi = s_seg_i[256 + ci];
                }
#pragma unroll
                for (int g8 = 0; g8 < 2; ++g8) {
                    float lk[8], lq[8], r[8];
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        const int u = g8 * 8 + w, t = 16 * tq + u;
                        const float kk = key_at(t, ci);
                        const float qq = query_at(t, ci);
                        fa *= al[u];
                        fi *= iv[u];
                        lk[w] = kk * fa;
                        lq[w] = qq * fa;
                        r[w] = kk * fi;
                    }
                    uint4 hi, lo;
                    const int tt = 16 * tq + g8 * 8;
                    split8(lk, hi, lo);
                    st16(sm, X_L_HI + chunk_mn(tt, ci, 1024, 2048), hi);
                    st16(sm, X_L_LO + chunk_mn(tt, ci, 1024, 2048), lo);
                    split8(lq, hi, lo);
                    st16(sm, X_L_HI + chunk_mn(64 + tt, ci, 1024, 2048), hi);
                    st16(sm, X_L_LO + chunk_mn(64 + tt, ci, 1024, 2048), lo);
                    split8(r, hi, lo);
                    st16(sm, X_R_HI + chunk_mn(tt, ci, 1024, 1024), hi);
                    st16(sm, X_R_LO + chunk_mn(tt, ci, 1024, 1024), lo);
                }
            }
            fence_async_smem();
            fence_before();
            __syncthreads();
            fence_after();
            // ---- MMA 1: [A; P] = [L_k; L_q] R^T: L_hi [R_hi; R_lo]^T (N = 128) + L_lo R_hi^T
            if (tid == 0) {
                const uint32_t id2 = idesc_bf16(128, 128, true, true, false);
                const uint32_t id1 = idesc_bf16(128, 64, true, true, false);
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma(tmem + TM_AP, desc_mn4(sb4 + X_L_HI / 16, 1024, 2048, s),
                        desc_mn4(sb4 + X_R_HI / 16, 16384, 1024, s), id2, s != 0);
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma(tmem + TM_AP, desc_mn4(sb4 + X_L_LO / 16, 1024, 2048, s),
                        desc_mn4(sb4 + X_R_HI / 16, 16384, 1024, s), id1, 1u);
                commit(mbar);
            }
            // ---- state pass (overlaps MMA 1): S_j -> snapshot, bf16 hi/lo A operand in TMEM,
            //      decay by e^{G_63}
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {  // 16 of this warp's 32 columns at a time
                const int col0 = cq * 32 + 16 * hh;
                float v[16];
                ld16(tl + TM_S + col0, v);
                for (int m = 0; m < p.M; ++m) {
                    if (s_trk[m] != j) continue;
                    const size_t snap = state_elem((int64_t)n * p.M + m, H, h) + (size_t)row * kD + col0;
#pragma unroll
                    for (int q4 = 0; q4 < 16; q4 += 4)
                        state_store4(p.track_state, snap + q4,
                                     make_float4(v[q4], v[q4 + 1], v[q4 + 2], v[q4 + 3]), p.st);
                }
                uint32_t sh[8], sl[8];
#pragma unroll
                for (int q2 = 0; q2 < 8; ++q2) split2(v[2 * q2], v[2 * q2 + 1], sh[q2], sl[q2]);
                st8u(tl + TM_SA_HI + cq * 16 + 8 * hh, sh);
                st8u(tl + TM_SA_LO + cq * 16 + 8 * hh, sl);
#pragma unroll
                for (int q = 0; q < 16; ++q) v[q] *= s_gam[col0 + q];
                st16f(tl + TM_S + col0, v);
            }
            wait_st();
            const bool ok1 = mbar_wait(mbar, phase, kWaitLimit);
            phase ^= 1;
            fence_after();
            if (__syncthreads_or(!ok1)) {
                timed_out = true;
                break;
            }

            // ---- A -> N = Diag(beta) A (strict lower, stored transposed: Nt[s][t] = N[t][s]),
            //      P -> bf16 operand (lower incl. diagonal)
            {
                float v[16], v2[16];
                ld16(tl + TM_AP + cq * 16, v);
                ld16(tl + TM_AP + 64 + cq * 16, v2);
#pragma unroll
                for (int q = 0; q < 16; ++q) v[q] += v2[q];
                float* Nt = reinterpret_cast<float*>(sm + X_N);
                if (quarter < 2) {
                    const int t = row;
                    const float bt = s_beta[t];
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int s = cq * 16 + q;
                        Nt[s * NLD + t] = s < t ? bt * v[q] : 0.f;
                    }
                } else {
                    const int t = row - 64;
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int s = cq * 16 + q;
                        if (s > t) v[q] = 0.f;
                    }
#pragma unroll
                    for (int c8 = 0; c8 < 2; ++c8) {
                        if constexpr (kBf16Out) {
                            st16(sm, X_P + chunk_k(t, cq * 16 + 8 * c8, 64), pack8(v + 8 * c8));
                        } else {
                            uint4 hi, lo;
                            split8(v + 8 * c8, hi, lo);
                            st16(sm, X_P + chunk_k(t, cq * 16 + 8 * c8, 64), hi);
                            st16(sm, X_P_LO + chunk_k(t, cq * 16 + 8 * c8, 64), lo);
                        }
                    }
                }
            }
            __syncthreads();
            // ---- T = (I + N)^-1 (unit lower triangular): 16x16 diagonal blocks by forward
            //      substitution, then the off-diagonal blocks by block substitution
            {
                const float* Nt = reinterpret_cast<const float*>(sm + X_N);
                float* Tm = reinterpret_cast<float*>(sm + X_T);
                if (tid < 64) {
                    // column jc of the inverse of diagonal block b: x = e_jc, then for each s
                    // (final from here on) x[r] -= N[r][s] x[s] for r > s
                    const int b = tid >> 4, jc = tid & 15, o = 16 * b;
                    float x[16];
#pragma unroll
                    for (int r = 0; r < 16; ++r) x[r] = (r == jc) ? 1.f : 0.f;
#pragma unroll
                    for (int s = 0; s < 15; ++s) {
                        float nr[16];
#pragma unroll
                        for (int r4 = (s + 1) / 4; r4 < 4; ++r4) {
                            const float4 n4 = *reinterpret_cast<const float4*>(&Nt[(o + s) * NLD + o + 4 * r4]);
                            nr[4 * r4] = n4.x;
                            nr[4 * r4 + 1] = n4.y;
                            nr[4 * r4 + 2] = n4.z;
                            nr[4 * r4 + 3] = n4.w;
                        }
                        const float xs = x[s];
#pragma unroll
                        for (int r = s + 1; r < 16; ++r) x[r] = fmaf(-nr[r], xs, x[r]);
                    }
#pragma unroll
                    for (int r = 0; r < 16; ++r) Tm[(o + r) * NLD + o + jc] = x[r];
                } else if (tid < 64 + 256) {
                    // the blocks above the diagonal pairs, (0,1) and (2,3), are zero
                    const int e = tid - 64, r = e >> 4, c = e & 15;
                    Tm[r * NLD + 16 + c] = 0.f;
                    Tm[(32 + r) * NLD + 48 + c] = 0.f;
                }
                __syncthreads();
                // level 1: T[a][a-1] = -T_aa N[a][a-1] T_{a-1,a-1}, a in {1, 3}; a thread owns
                // row r and 4 adjacent columns of one 16x16 block
                float* Y1 = reinterpret_cast<float*>(sm + X_Y1);  // [2][16][20]
                const int w1 = tid >> 6, r1 = (tid & 63) >> 2, c1 = (tid & 3) * 4;
                const int oa = 32 * w1 + 16, ob = 32 * w1;
                if (tid < 128) {
                    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int s = 0; s < 16; ++s) {
                        const float nv = Nt[(ob + s) * NLD + oa + r1];
                        const float4 tv = *reinterpret_cast<const float4*>(&Tm[(ob + s) * NLD + ob + c1]);
                        y.x = fmaf(nv, tv.x, y.x);
                        y.y = fmaf(nv, tv.y, y.y);
                        y.z = fmaf(nv, tv.z, y.z);
                        y.w = fmaf(nv, tv.w, y.w);
                    }
                    *reinterpret_cast<float4*>(&Y1[(w1 * 16 + r1) * 20 + c1]) = y;
                }
                __syncthreads();
                if (tid < 128) {
                    float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int s = 0; s < 16; ++s) {
                        const float tv = Tm[(oa + r1) * NLD + oa + s];
                        const float4 yv = *reinterpret_cast<const float4*>(&Y1[(w1 * 16 + s) * 20 + c1]);
                        z.x = fmaf(tv, yv.x, z.x);
                        z.y = fmaf(tv, yv.y, z.y);
                        z.z = fmaf(tv, yv.z, z.z);
                        z.w = fmaf(tv, yv.w, z.w);
                    }
                    *reinterpret_cast<float4*>(&Tm[(oa + r1) * NLD + ob + c1]) =
                        make_float4(-z.x, -z.y, -z.z, -z.w);
                }
                __syncthreads();
                // level 2: T[32:64, 0:32] = -T[32:64, 32:64] (N[32:64, 0:32] T[0:32, 0:32]).
                // First product: warp = 4-column group c2, lane = row; T[0:32, 0:32] is lower
                // triangular, so the sum starts at u = c2.
                float* Y2 = reinterpret_cast<float*>(sm + X_Y2);  // [32][36]
                if (tid < 256) {
                    const int c2 = 4 * warp;
                    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
                    for (int u = c2; u < 32; ++u) {
                        const float nv = Nt[u * NLD + 32 + lane];
                        const float4 tv = *reinterpret_cast<const float4*>(&Tm[u * NLD + c2]);
                        y.x = fmaf(nv, tv.x, y.x);
                        y.y = fmaf(nv, tv.y, y.y);
                        y.z = fmaf(nv, tv.z, y.z);
                        y.w = fmaf(nv, tv.w, y.w);
                    }
                    *reinterpret_cast<float4*>(&Y2[lane * 36 + c2]) = y;
                }
                __syncthreads();
                if (tid < 256) {
                    const int r = tid >> 3, c = (tid & 7) * 4;
                    float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
                    for (int s = 0; s < 32; ++s) {
                        const float tv = Tm[(32 + r) * NLD + 32 + s];
                        const float4 yv = *reinterpret_cast<const float4*>(&Y2[s * 36 + c]);
                        z.x = fmaf(tv, yv.x, z.x);
                        z.y = fmaf(tv, yv.y, z.y);
                        z.z = fmaf(tv, yv.z, z.z);
                        z.w = fmaf(tv, yv.w, z.w);
                    }
                    *reinterpret_cast<float4*>(&Tm[(32 + r) * NLD + c]) = make_float4(-z.x, -z.y, -z.z, -z.w);
                }
                __syncthreads();
                // T_b = T Diag(beta) -> bf16 hi/lo operand [t][s] (lower triangle only)
                {
                    const int t = tid >> 3, s0 = (tid & 7) * 8;
                    float x[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const int s = s0 + q;
                        x[q] = s <= t ? Tm[t * NLD + s] * s_beta[s] : 0.f;
                    }
                    uint4 hi, lo;
                    split8(x, hi, lo);
                    st16(sm, OFF_TB_HI + chunk_k(t, s0, 64), hi);
                    st16(sm, OFF_TB_LO + chunk_k(t, s0, 64), lo);
                }
            }
            __syncthreads();
            // ---- KG = k e^{G} (A, [i][s]), QG = q e^{G} (B, MN-major), KT = k e^{G_63 - G} ([i][s])
            {
                const float a0 = s_seg_a[ci], a1 = s_seg_a[128 + ci], a2 = s_seg_a[256 + ci],
                            a3 = s_seg_a[384 + ci];
                // e^{G_t}: running product from the chunk start; e^{G_63 - G_t}: product over (t, 63]
                float fw = tq == 0 ? 1.f : tq == 1 ? a0 : tq == 2 ? a0 * a1 : (a0 * a1) * a2;
                float bw = tq == 3 ? 1.f : tq == 2 ? a3 : tq == 1 ? a2 * a3 : a1 * (a2 * a3);
                uint32_t kgh[8], kgl[8];  // KG row ci, tokens 16*tq.., packed bf16 pairs
#pragma unroll
                for (int c8 = 0; c8 < 2; ++c8) {
                    float kg[8], qg[8];
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        const int u = 8 * c8 + w, t = 16 * tq + u;
                        fw *= al[u];
                        kg[w] = key_at(t, ci) * fw;
                        qg[w] = query_at(t, ci) * fw;
                    }
                    const int s0 = 16 * tq + 8 * c8;
                    uint4 hi, lo;
                    split8(kg, hi, lo);
                    kgh[4 * c8] = hi.x; kgh[4 * c8 + 1] = hi.y; kgh[4 * c8 + 2] = hi.z; kgh[4 * c8 + 3] = hi.w;
                    kgl[4 * c8] = lo.x; kgl[4 * c8 + 1] = lo.y; kgl[4 * c8 + 2] = lo.z; kgl[4 * c8 + 3] = lo.w;
                    if constexpr (kBf16Out) {
                        st16(sm, X_QG + chunk_mn(s0, ci, 1024, 1024), pack8(qg));
                    } else {
                        split8(qg, hi, lo);
                        st16(sm, X_QG + chunk_mn(s0, ci, 1024, 1024), hi);
                        st16(sm, OFF_QG_LO + chunk_mn(s0, ci, 1024, 1024), lo);
                    }
                }
#pragma unroll
                for (int c8 = 1; c8 >= 0; --c8) {
                    float kt[8];
#pragma unroll
                    for (int w = 7; w >= 0; --w) {
                        const int u = 8 * c8 + w, t = 16 * tq + u;
                        kt[w] = key_at(t, ci) * bw;
                        bw *= al[u];
                    }
                    const int s0 = 16 * tq + 8 * c8;
                    uint4 hi, lo;
                    split8(kt, hi, lo);
                    st16(sm, X_KT_HI + chunk_k(ci, s0, 128), hi);
                    st16(sm, X_KT_LO + chunk_k(ci, s0, 128), lo);
                }
                st8u(tl + TM_KG_HI + tq * 8, kgh);  // lane ci of this warp's quarter
                st8u(tl + TM_KG_LO + tq * 8, kgl);
                wait_st();
            }
            fence_async_smem();
            fence_before();
            __syncthreads();
            fence_after();
            if (more) {
                prefetch_qkg(j + 1);  // the raw q, k, g tiles of this chunk are consumed
                cp_async_commit();
            }
            // ---- MMA 2: W^T = KG T_b^T (into the O columns), U~^T = V^T [T_b hi; T_b lo]^T
            //      (N = 128, into [U_a | U_b])
            if (tid == 0) {
                const uint32_t idk = idesc_bf16(128, 64, false, false, false);
                const uint32_t idv = idesc_bf16(128, 128, true, false, false);
#pragma unroll
                for (int pass = 0; pass < 3; ++pass) {
                    const uint32_t a = tmem + (pass == 2 ? TM_KG_LO : TM_KG_HI);
                    const uint32_t b = sb4 + (pass == 1 ? OFF_TB_LO : OFF_TB_HI) / 16;
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        mma_ta(tmem + TM_O, a + 8 * s, desc_k4(b, 64, s), idk, (pass | s) != 0);
                }
                commit(mbar);  // W^T only: U~^T (below) keeps running while W is extracted
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma(tmem + TM_UA, desc_mn4(sb4 + v_cur / 16, 8192, 1024, s),
                        desc_k4(sb4 + OFF_TB_HI / 16, 128, s), idv, s != 0);
            }
            const bool ok2 = mbar_wait(mbar, phase, kWaitLimit);
            phase ^= 1;
            fence_after();
            if (__syncthreads_or(!ok2)) {
                timed_out = true;
                break;
            }
            // ---- W^T (lanes i, columns t) -> -W operand (B, MN-major [i][t]) hi/lo; the O
            //      columns are then cleared for MMA 3 to accumulate into
            {
                float v[16];
                ld16(tl + TM_O + cq * 16, v);
#pragma unroll
                for (int q = 0; q < 16; ++q) v[q] = -v[q];
#pragma unroll
                for (int c8 = 0; c8 < 2; ++c8) {
                    uint4 hi, lo;
                    split8(v + 8 * c8, hi, lo);
                    const int t = cq * 16 + 8 * c8;
                    st16(sm, X_W_HI + chunk_mn(t, row, 1024, 1024), hi);
                    st16(sm, X_W_LO + chunk_mn(t, row, 1024, 1024), lo);
                }
#pragma unroll
                for (int q = 0; q < 16; ++q) v[q] = 0.f;
                st16f(tl + TM_O + cq * 16, v);
                wait_st();
            }
            fence_async_smem();
            fence_before();
            __syncthreads();
            fence_after();
            // ---- MMA 3: [O | U_a | U_b] += S_hi^T [QG; -W_hi; -W_lo]^T (N = 192),
            //      [O | U_a] += S_lo^T [QG; -W_hi]^T (N = 128); fp32 outputs also S_hi^T QG_lo^T.
            //      U^T = U~^T - S^T W^T = U_a + U_b.  The commit also covers MMA 2's reads of V.
            if (tid == 0) {
                const uint32_t id3 = idesc_bf16(128, 192, false, true, false);
                const uint32_t id2 = idesc_bf16(128, 128, false, true, false);
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_ta(tmem + TM_O, tmem + TM_SA_HI + 8 * s, desc_mn4(sb4 + X_QG / 16, 16384, 1024, s),
                           id3, 1u);
#pragma unroll
                for (int s = 0; s < 8; ++s)
                    mma_ta(tmem + TM_O, tmem + TM_SA_LO + 8 * s, desc_mn4(sb4 + X_QG / 16, 16384, 1024, s),
                           id2, 1u);
                if constexpr (!kBf16Out) {
                    const uint32_t id1 = idesc_bf16(128, 64, false, true, false);
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        mma_ta(tmem + TM_O, tmem + TM_SA_HI + 8 * s,
                               desc_mn4(sb4 + OFF_QG_LO / 16, 16384, 1024, s), id1, 1u);
                }
                commit(mbar);
            }
            const bool ok3 = mbar_wait(mbar, phase, kWaitLimit);
            phase ^= 1;
            fence_after();
            if (__syncthreads_or(!ok3)) {
                timed_out = true;
                break;
            }
            // ---- U^T (lanes c, columns s) -> bf16 hi/lo A operand in TMEM
            {
                float v[16], v2[16];
                ld16(tl + TM_UA + cq * 16, v);
                ld16(tl + TM_UB + cq * 16, v2);
#pragma unroll
                for (int q = 0; q < 16; ++q) v[q] += v2[q];
                uint32_t uh[8], ul[8];
#pragma unroll
                for (int q2 = 0; q2 < 8; ++q2) split2(v[2 * q2], v[2 * q2 + 1], uh[q2], ul[q2]);
                st8u(tl + TM_U_HI + cq * 8, uh);
                st8u(tl + TM_U_LO + cq * 8, ul);
                wait_st();
            }
            fence_before();
            __syncthreads();
            fence_after();
            // ---- MMA 4: [S | O] += U_hi^T [KT_hi; P]^T (N = 192); then the rest of the state
            //      update, S^T += U_lo^T KT_hi + U_hi^T KT_lo, completes in the background
            if (tid == 0) {
                const uint32_t id3 = idesc_bf16(128, 192, false, false, false);
                const uint32_t id2 = idesc_bf16(128, 128, false, false, false);
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_ta(tmem + TM_S, tmem + TM_U_HI + 8 * s, desc_k4(sb4 + X_KT_HI / 16, 192, s), id3, 1u);
                if constexpr (!kBf16Out) {
                    const uint32_t id1 = idesc_bf16(128, 64, false, false, false);
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        mma_ta(tmem + TM_S, tmem + TM_U_LO + 8 * s, desc_k4(sb4 + X_KT_HI / 16, 192, s), id3,
                               1u);
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        mma_ta(tmem + TM_O, tmem + TM_U_HI + 8 * s, desc_k4(sb4 + X_P_LO / 16, 64, s), id1, 1u);
                }
                commit(mbar);  // the outputs
                if constexpr (kBf16Out) {
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        mma_ta(tmem + TM_S, tmem + TM_U_LO + 8 * s, desc_k4(sb4 + X_KT_HI / 16, 128, s), id2,
                               1u);
                }
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_ta(tmem + TM_S, tmem + TM_U_HI + 8 * s, desc_k4(sb4 + X_KT_LO / 16, 128, s), id2, 1u);
                commit(mbar_s);
            }
            pending_s = true;
            const bool ok4 = mbar_wait(mbar, phase, kWaitLimit);
            phase ^= 1;
            fence_after();
            if (__syncthreads_or(!ok4)) {
                timed_out = true;
                break;
            }
            // ---- O^T (lanes c, columns t) -> out[t][h][c]
            {
                float v[16];
                ld16(tl + TM_O + cq * 16, v);
                if constexpr (kBf16Out) {
                    // through shared memory (the T_b region, free now) for 16-byte row stores
                    __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(sm + OFF_TB_HI);
#pragma unroll
                    for (int q = 0; q < 16; ++q)
                        ob[(cq * 16 + q) * kD + row] = __float2bfloat16_rn(v[q]);
                    __syncthreads();
#pragma unroll
                    for (int it = tid; it < 64 * 16; it += kThreads) {
                        const int t = it >> 4, ch = it & 15;
                        if (t < Lc)
                            *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) +
                                                      ((size_t)(c0 + t) * H + h) * kD + ch * 8) =
                                *reinterpret_cast<const uint4*>(sm + OFF_TB_HI + t * 256 + ch * 16);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int t = cq * 16 + q;
                        if (t < Lc) store1<false>(p.out, ((size_t)(c0 + t) * H + h) * kD + row, v[q]);
                    }
                }
            }
        } else {
            // ---- fallback: this chunk token by token on CUDA cores
            float* alpha = reinterpret_cast<float*>(sm + X_ALPHA);
#pragma unroll
            for (int u = 0; u < 16; ++u) alpha[(16 * tq + u) * kD + ci] = al[u];
            fence_before();
            __syncthreads();
            fence_after();
            {
                // thread (row c, column quarter) keeps 32 state columns in registers; the four
                // partial row dot products meet in shared memory
                float* red = reinterpret_cast<float*>(sm + X_RED);  // [2 dots][4 quarters][128]
                const int c = row;
                float sv[32];
                ld32(tl + TM_S + cq * 32, sv);
                for (int m = 0; m < p.M; ++m) {
                    if (s_trk[m] != j) continue;
                    const size_t snap = state_elem((int64_t)n * p.M + m, H, h) + (size_t)c * kD + cq * 32;
#pragma unroll
                    for (int q4 = 0; q4 < 32; q4 += 4)
                        state_store4(p.track_state, snap + q4,
                                     make_float4(sv[q4], sv[q4 + 1], sv[q4 + 2], sv[q4 + 3]), p.st);
                }
                for (int t = 0; t < Lc; ++t) {
                    float d1 = 0.f;
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        const int i = cq * 32 + q;
                        sv[q] *= alpha[t * kD + i];
                        d1 = fmaf(sv[q], key_at(t, i), d1);
                    }
                    red[cq * 128 + c] = d1;
                    __syncthreads();
                    d1 = (red[c] + red[128 + c]) + (red[256 + c] + red[384 + c]);
                    const float vt = bf16_at(sm, v_cur + chunk_mn(c & ~7, t, 8192, 1024) + (c & 7) * 2);
                    const float uu = s_beta[t] * (vt - d1);
                    float o = 0.f;
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        const int i = cq * 32 + q;
                        sv[q] = fmaf(uu, key_at(t, i), sv[q]);
                        o = fmaf(sv[q], query_at(t, i), o);
                    }
                    red[512 + cq * 128 + c] = o;
                    __syncthreads();
                    if (cq == 0)
                        store1<kBf16Out>(p.out, ((size_t)(c0 + t) * H + h) * kD + c,
                                         (red[512 + c] + red[640 + c]) + (red[768 + c] + red[896 + c]));
                }
                st32(tl + TM_S + cq * 32, sv);
                wait_st();
            }
            fence_before();
            __syncthreads();
            fence_after();
            if (more) {
                prefetch_qkg(j + 1);
                cp_async_commit();
            }
        }
    }
    cp_async_wait_all();

    if (pending_s && !timed_out) {
        if (!mbar_wait(mbar_s, phase_s, kWaitLimit)) timed_out = true;
        pending_s = false;
    }
    fence_before();
    timed_out = __syncthreads_or(timed_out);
    fence_after();
    if (timed_out) {
        if (tid == 0) report(p.dev_status, KDA_DEV_TIMEOUT);
        // give in-flight MMAs a bounded chance to drain before TMEM is released: the last
        // phase waited on of each barrier (it may be the one that timed out; a wait on a
        // completed phase returns at once) and a state update issued but not yet waited on
        mbar_wait(mbar, phase ^ 1u, kWaitLimit);
        mbar_wait(mbar_s, phase_s ^ 1u, kWaitLimit);
        if (pending_s) mbar_wait(mbar_s, phase_s, kWaitLimit);
    } else if (fin >= 0) {
        const size_t SD = state_elem(fin, H, h) + (size_t)row * kD;
        const int col0 = cq * 32;
        float v[32];
        ld32(tl + TM_S + col0, v);
#pragma unroll
        for (int q4 = 0; q4 < 32; q4 += 4)
            state_store4(p.pool, SD + col0 + q4, make_float4(v[q4], v[q4 + 1], v[q4 + 2], v[q4 + 3]),
                         p.st);
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

// Longest sequence first, so that the longest serial chains start in the first wave.
__global__ void __launch_bounds__(1024) prefill_order_kernel(const int32_t* __restrict__ cu, int N,
                                                              int32_t* __restrict__ order) {
    for (int n = threadIdx.x; n < N; n += blockDim.x) {
        const int Ln = cu[n + 1] - cu[n];
        int rank = 0;
        for (int m = 0; m < N; ++m) {
            const int Lm = cu[m + 1] - cu[m];
            rank += (Lm > Ln) || (Lm == Ln && m < n);
        }
        order[rank] = n;
    }
}

}  // namespace

bool prefill_tc_supported(const PrefillArgs& p, bool bf16_in) {
    return bf16_in && p.M <= kTrackTc;
}

size_t prefill_tc_workspace(int32_t N) {
    return N > 0 && N <= kMaxOrderN ? (size_t)((N + 3) / 4) * 16 : 0;
}

void launch_prefill_tc(const PrefillArgs& p, bool bf16_out, void* workspace, size_t ws_bytes,
                       cudaStream_t s) {
    int32_t* order = nullptr;
    const size_t need = prefill_tc_workspace(p.N);
    if (workspace && need > 0 && ws_bytes >= need) {
        order = static_cast<int32_t*>(workspace);
        prefill_order_kernel<<<1, 1024, 0, s>>>(p.cu_seqlens, p.N, order);
    }
    const unsigned grid = (unsigned)(p.N * p.H);
    if (bf16_out) {
        cudaFuncSetAttribute(prefill_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES);
        prefill_tc_kernel<true><<<grid, kThreads, SMEM_BYTES, s>>>(p, order);
    } else {
        cudaFuncSetAttribute(prefill_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES);
        prefill_tc_kernel<false><<<grid, kThreads, SMEM_BYTES, s>>>(p, order);
    }
}

}  // namespace kda
