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
// The snapshot of chunk j (the state after j*64 tokens of the sequence, SGLang
// PR 34820 page, the fp32 track-state snapshot) is written from the fp32 TMEM
// accumulator when chunk j starts.
#include "kda_common.cuh"
#include "kda_host.h"
#include "prefill.h"
#include "umma.cuh"

namespace kda {
namespace {

using namespace umma;

constexpr int kThreads = 256;
constexpr int kTrackTc = 512;  // snapshot requests per sequence handled by this kernel

// shared memory map (bytes from a 1024-aligned base)
constexpr uint32_t OFF_ST_HI = 0;  // A: S^T [c][i], K-major, 128 rows, K = 128; before the
constexpr uint32_t OFF_ST_LO = 32768;  // state pass the raw q, k, g tiles of the chunk (row-major)
constexpr uint32_t OFF_X = 65536;  // 96 KiB reused by the chunk phases:
//   fallback alpha (fp32 [64][128]), dot scratch     X+0, X+32K
//   L hi/lo (A, MN-major, M = 128, K = 128)          X+0,  X+32K
//   R hi/lo (B, MN-major, N = 64,  K = 128)          X+64K, X+80K
//   N, T (fp32 [64][68]) and solve temporaries       X+0 .. X+41K
//   KG hi/lo (A, K-major [i][s]), QG (B, MN-major),
//   KT hi/lo (B, K-major [i][s]), QG lo              X+0, X+16K, X+32K, X+48K, X+64K, X+80K
//   W hi/lo (B, MN-major [i][t])                     X+0, X+16K
//   UT hi/lo (A, K-major [c][s])                     X+0, X+16K
constexpr uint32_t OFF_V = OFF_X + 98304;        // A: V, MN-major (c atoms 8 KiB apart, s groups 1 KiB)
constexpr uint32_t OFF_TB_HI = OFF_V + 16384;    // B: T_b [t][s], K-major, 64 rows
constexpr uint32_t OFF_TB_LO = OFF_TB_HI + 8192;
constexpr uint32_t OFF_P = OFF_TB_LO + 8192;     // B: P [t][s], K-major, 64 rows
constexpr uint32_t OFF_P_LO = OFF_P + 8192;      // P lo (fp32 outputs only)
constexpr uint32_t OFF_MISC = OFF_P_LO + 8192;
constexpr uint32_t MISC_BYTES = 8192;
constexpr uint32_t SMEM_BYTES = OFF_MISC + MISC_BYTES + 1024;  // + alignment slack

constexpr uint32_t RAW_Q = OFF_ST_HI, RAW_K = OFF_ST_HI + 16384, RAW_G = OFF_ST_HI + 32768;
constexpr uint32_t X_ALPHA = OFF_X, X_RED = OFF_X + 32768;
constexpr uint32_t X_L_HI = OFF_X, X_L_LO = OFF_X + 32768, X_R_HI = OFF_X + 65536,
                   X_R_LO = OFF_X + 81920;
constexpr uint32_t X_N = OFF_X, X_T = OFF_X + 17408, X_Y1 = OFF_X + 34816, X_Y2 = OFF_X + 37376;
constexpr uint32_t X_KG_HI = OFF_X, X_KG_LO = OFF_X + 16384, X_QG = OFF_X + 32768,
                   X_KT_HI = OFF_X + 49152, X_KT_LO = OFF_X + 65536, X_QG_LO = OFF_X + 81920;
constexpr uint32_t X_W_HI = OFF_X, X_W_LO = OFF_X + 16384;
constexpr uint32_t X_UT_HI = OFF_X, X_UT_LO = OFF_X + 16384;
constexpr int NLD = 68;  // fp32 row stride of the N / T matrices

// TMEM columns
constexpr uint32_t TM_S = 0, TM_AP = 128, TM_WT = 192, TM_UT = 256, TM_OT = 320;
constexpr uint32_t TM_COLS = 512;

constexpr uint32_t kWaitLimit = 1u << 22;    // polls; a healthy MMA batch completes in microseconds
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
    float* s_beta = reinterpret_cast<float*>(sm + OFF_MISC);  // 64
    float* s_gam = s_beta + 64;                               // 128
    float* s_tot0 = s_gam + 128;                              // 128
    float* s_tot1 = s_tot0 + 128;                             // 128
    int* s_trk = reinterpret_cast<int*>(s_tot1 + 128);        // kTrackTc
    uint64_t* s_mbar = reinterpret_cast<uint64_t*>(s_trk + kTrackTc);  // [0]: MMA batches, [1]: state update
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(s_mbar + 2);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3;   // TMEM lane quarter this warp may access
    const int colhalf = warp >> 2;  // which column half this warp takes in TMEM passes
    const int row = quarter * 32 + lane;
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

    // ---- TMEM and the MMA completion barrier
    if (warp == 0) tmem_alloc(smem_u32(s_tmem), TM_COLS);
    if (tid == 0) {
        mbar_init(smem_u32(s_mbar), 1);
        mbar_init(smem_u32(s_mbar + 1), 1);
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

    // ---- initial state into TMEM (row c = S^T row, this thread's 64 columns)
    {
        const float* S0 = init >= 0 ? p.pool + ((size_t)init * H + h) * (kD * kD) : nullptr;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int col0 = colhalf * 64 + cc * 32;
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                float4 x = S0 ? reinterpret_cast<const float4*>(S0 + (size_t)row * kD + col0 + j)[0]
                              : make_float4(0.f, 0.f, 0.f, 0.f);
                v[j] = x.x;
                v[j + 1] = x.y;
                v[j + 2] = x.z;
                v[j + 3] = x.w;
            }
            st32(tl + TM_S + col0, v);
        }
        wait_st();
    }

    const int ci = tid & 127, hf = tid >> 7;  // channel-pass mapping: key channel, half chunk
    bool timed_out = false;
    const __nv_bfloat16* gq = static_cast<const __nv_bfloat16*>(p.q);
    const __nv_bfloat16* gk = static_cast<const __nv_bfloat16*>(p.k);
    const __nv_bfloat16* gv = static_cast<const __nv_bfloat16*>(p.v);
    const __nv_bfloat16* gg = static_cast<const __nv_bfloat16*>(p.gate_raw);

    // Raw tiles of chunk jj arrive by cp.async: q, k, g row-major into the
    // S-operand region (free from MMA 3 of the previous chunk until the state
    // pass), v as the MN-major MMA operand (free after MMA 2).  Rows past the
    // sequence are zero-filled.
    auto prefetch_qkg = [&](int jj) {
        const int cn = t0 + jj * kChunk, ln = min(kChunk, t1 - cn);
#pragma unroll 4
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
#pragma unroll 4
        for (int it = tid; it < 64 * 16; it += kThreads) {
            const int t = it >> 4, ch = it & 15;
            const bool ok = t < ln;
            const size_t e = ok ? ((size_t)(cn + t) * H + h) * kD + ch * 8 : 0;
            cp_async16(sb + OFF_V + chunk_mn(ch * 8, t, 8192, 1024), gv + e, ok ? 16u : 0u);
        }
    };
    // raw beta of chunk jj (activated when the chunk starts, so the load is never waited on
    // early); -inf marks padding rows, whose beta is 0
    auto load_beta = [&](int jj) {
        const int cn = t0 + jj * kChunk, ln = min(kChunk, t1 - cn);
        return tid < ln ? Act<true>::load1(p.beta_raw, (size_t)(cn + tid) * H + h) : -INFINITY;
    };
    float beta_next = 0.f;
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
        if (pending_s) {  // the previous state update still reads UT / KT and writes S
            const bool ok = mbar_wait(mbar_s, phase_s, kWaitLimit);
            phase_s ^= 1;
            pending_s = false;
            if (!ok) timed_out = true;
        }
        if (tid < 64) s_beta[tid] = tid < Lc ? beta_act(beta_next, p.flags) : 0.f;
        fence_before();
        if (__syncthreads_or(timed_out)) {
            timed_out = true;
            break;
        }
        fence_after();
        if (tid < 64 && more) beta_next = load_beta(j + 1);  // lands during this chunk

        // ---- channel pass: this thread's channel ci over tokens 32*hf .. 32*hf+31
        float al[32], iv[32];
#pragma unroll
        for (int u = 0; u < 32; ++u) {
            const int t = 32 * hf + u;
            const float x = bf16_at(sm, RAW_G + t * 256 + ci * 2);
            if (t < Lc) {
                if (p.flags & KDA_GATE_LOG) {
                    al[u] = __expf(x);
                    iv[u] = __expf(-x);
                } else {
                    iv[u] = 1.f + __expf(x);  // 1/alpha = 1 + e^x
                    al[u] = __fdividef(1.f, iv[u]);
                }
            } else {
                al[u] = 1.f;
                iv[u] = 1.f;
            }
        }
        bool bad;
        {
            // largest factor >= 1 this half uses: prod of 1/alpha over (0, 31] (half 0) or [32, 63]
            float m = 1.f;
#pragma unroll
            for (int u = 0; u < 32; ++u)
                if (hf == 1 || u > 0) m *= iv[u];
            bad = !(m <= kFactorMax);
        }
        const int fallback = __syncthreads_or(bad);

        if (!fallback) {
            // ---- L = [k; q] e^{G_t - G_31}, R = k e^{G_31 - G_s} (half 0: backward from 31;
            //      half 1: forward from 32), half totals for e^{G_31} and e^{G_63 - G_31}
            if (hf == 0) {
                float sa = 1.f, si = 1.f;  // prod over (u, 31] of alpha and of 1/alpha
#pragma unroll
                for (int g8 = 3; g8 >= 0; --g8) {
                    float lk[8], lq[8], r[8];
#pragma unroll
                    for (int w = 7; w >= 0; --w) {
                        const int u = g8 * 8 + w;
                        const float kk = bf16_at(sm, RAW_K + u * 256 + ci * 2);
                        const float qq = bf16_at(sm, RAW_Q + u * 256 + ci * 2) * p.scale;
                        lk[w] = kk * si;
                        lq[w] = qq * si;
                        r[w] = kk * sa;
                        sa *= al[u];
                        si *= iv[u];
                    }
                    uint4 hi, lo;
                    const int tt = g8 * 8;
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
                s_tot0[ci] = sa;  // e^{G_31}
            } else {
                float fa = 1.f, fi = 1.f;  // prod over [32, 32+u] of alpha and of 1/alpha
#pragma unroll
                for (int g8 = 0; g8 < 4; ++g8) {
                    float lk[8], lq[8], r[8];
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        const int u = g8 * 8 + w;
                        const float kk = bf16_at(sm, RAW_K + (32 + u) * 256 + ci * 2);
                        const float qq = bf16_at(sm, RAW_Q + (32 + u) * 256 + ci * 2) * p.scale;
                        fa *= al[u];
                        fi *= iv[u];
                        lk[w] = kk * fa;
                        lq[w] = qq * fa;
                        r[w] = kk * fi;
                    }
                    uint4 hi, lo;
                    const int tt = 32 + g8 * 8;
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
                s_tot1[ci] = fa;  // e^{G_63 - G_31}
            }
            fence_async_smem();
            fence_before();
            __syncthreads();
            fence_after();
            // ---- MMA 1: [A; P] = [L_k; L_q] R^T
            if (tid == 0) {
                const uint32_t id = idesc_bf16(128, 64, true, true, false);
#pragma unroll
                for (int pass = 0; pass < 3; ++pass) {
                    const uint32_t a = sb + (pass == 2 ? X_L_LO : X_L_HI);
                    const uint32_t b = sb + (pass == 1 ? X_R_LO : X_R_HI);
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        mma(tmem + TM_AP, desc_mn(a, 1024, 2048, s), desc_mn(b, 1024, 1024, s), id,
                            (pass | s) != 0);
                }
                commit(mbar);
            }
            if (hf == 0) s_gam[ci] = s_tot0[ci] * s_tot1[ci];
            const bool ok1 = mbar_wait(mbar, phase, kWaitLimit);
            phase ^= 1;
            fence_after();
            if (__syncthreads_or(!ok1)) {
                timed_out = true;
                break;
            }

            // ---- A -> N = Diag(beta) A (strict lower), P -> bf16 operand (lower incl. diagonal)
            {
                float v[32];
                ld32(tl + TM_AP + colhalf * 32, v);
                float* Nm = reinterpret_cast<float*>(sm + X_N);
                if (quarter < 2) {
                    const int t = row;
                    const float bt = s_beta[t];
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        const int s = colhalf * 32 + q;
                        Nm[t * NLD + s] = s < t ? bt * v[q] : 0.f;
                    }
                } else {
                    const int t = row - 64;
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        const int s = colhalf * 32 + q;
                        if (s > t) v[q] = 0.f;
                    }
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) {
                        if constexpr (kBf16Out) {
                            st16(sm, OFF_P + chunk_k(t, colhalf * 32 + 8 * c8, 64), pack8(v + 8 * c8));
                        } else {
                            uint4 hi, lo;
                            split8(v + 8 * c8, hi, lo);
                            st16(sm, OFF_P + chunk_k(t, colhalf * 32 + 8 * c8, 64), hi);
                            st16(sm, OFF_P_LO + chunk_k(t, colhalf * 32 + 8 * c8, 64), lo);
                        }
                    }
                }
            }
            __syncthreads();
            // ---- T = (I + N)^-1: 16x16 diagonal blocks, then block substitution
            {
                const float* Nm = reinterpret_cast<const float*>(sm + X_N);
                float* Tm = reinterpret_cast<float*>(sm + X_T);
                if (tid < 64) {
                    const int b = tid >> 4, jc = tid & 15, o = 16 * b;
                    float x[16];
#pragma unroll
                    for (int r = 0; r < 16; ++r) {
                        float acc = 0.f;
#pragma unroll
                        for (int s = 0; s < r; ++s) acc = fmaf(Nm[(o + r) * NLD + o + s], x[s], acc);
                        x[r] = (r == jc) ? 1.f : -acc;
                    }
#pragma unroll
                    for (int r = 0; r < 16; ++r) Tm[(o + r) * NLD + o + jc] = x[r];
                }
                __syncthreads();
                // level 1: T[a][a-1] = -D_a N[a][a-1] D_{a-1}, a in {1, 3}; a thread owns one
                // row r and 2 adjacent columns of one 16x16 block
                float* Y1 = reinterpret_cast<float*>(sm + X_Y1);  // [2][16][20]
                {
                    const int w = tid >> 7, e = tid & 127, r = e >> 3, c = (e & 7) * 2;
                    const int a = 2 * w + 1, oa = 16 * a, ob = 16 * (a - 1);
                    float y0 = 0.f, y1 = 0.f;
#pragma unroll
                    for (int s = 0; s < 16; ++s) {
                        const float nv = Nm[(oa + r) * NLD + ob + s];
                        const float2 tv = *reinterpret_cast<const float2*>(&Tm[(ob + s) * NLD + ob + c]);
                        y0 = fmaf(nv, tv.x, y0);
                        y1 = fmaf(nv, tv.y, y1);
                    }
                    *reinterpret_cast<float2*>(&Y1[(w * 16 + r) * 20 + c]) = make_float2(y0, y1);
                    // T is lower triangular: the blocks above the diagonal pairs are zero
                    Tm[(16 * (2 * w) + r) * NLD + 16 * (2 * w + 1) + c] = 0.f;
                    Tm[(16 * (2 * w) + r) * NLD + 16 * (2 * w + 1) + c + 1] = 0.f;
                    __syncthreads();
                    float z0 = 0.f, z1 = 0.f;
#pragma unroll
                    for (int s = 0; s < 16; ++s) {
                        const float tv = Tm[(oa + r) * NLD + oa + s];
                        const float2 yv = *reinterpret_cast<const float2*>(&Y1[(w * 16 + s) * 20 + c]);
                        z0 = fmaf(tv, yv.x, z0);
                        z1 = fmaf(tv, yv.y, z1);
                    }
                    *reinterpret_cast<float2*>(&Tm[(oa + r) * NLD + ob + c]) = make_float2(-z0, -z1);
                }
                __syncthreads();
                // level 2: T[32:64, 0:32] = -T[32:64, 32:64] (N[32:64, 0:32] T[0:32, 0:32]);
                // a thread owns one row r and 4 adjacent columns
                float* Y2 = reinterpret_cast<float*>(sm + X_Y2);  // [32][36]
                {
                    const int r = tid >> 3, c = (tid & 7) * 4;
                    float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
                    for (int u = 0; u < 32; ++u) {
                        const float nv = Nm[(32 + r) * NLD + u];
                        const float4 tv = *reinterpret_cast<const float4*>(&Tm[u * NLD + c]);
                        y.x = fmaf(nv, tv.x, y.x);
                        y.y = fmaf(nv, tv.y, y.y);
                        y.z = fmaf(nv, tv.z, y.z);
                        y.w = fmaf(nv, tv.w, y.w);
                    }
                    *reinterpret_cast<float4*>(&Y2[r * 36 + c]) = y;
                    __syncthreads();
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
#pragma unroll
                for (int it = tid; it < 64 * 8; it += kThreads) {
                    const int t = it >> 3, s0 = (it & 7) * 8;
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
                const float t0f = s_tot0[ci], t1f = s_tot1[ci];
                float fw = (hf == 0) ? 1.f : t0f;  // e^{G_t}: running product from the chunk start
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    float kg[8], qg[8];
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        const int u = 8 * c8 + w, t = 32 * hf + u;
                        fw *= al[u];
                        kg[w] = bf16_at(sm, RAW_K + t * 256 + ci * 2) * fw;
                        qg[w] = bf16_at(sm, RAW_Q + t * 256 + ci * 2) * p.scale * fw;
                    }
                    const int s0 = 32 * hf + 8 * c8;
                    uint4 hi, lo;
                    split8(kg, hi, lo);
                    st16(sm, X_KG_HI + chunk_k(ci, s0, 128), hi);
                    st16(sm, X_KG_LO + chunk_k(ci, s0, 128), lo);
                    if constexpr (kBf16Out) {
                        st16(sm, X_QG + chunk_mn(s0, ci, 1024, 1024), pack8(qg));
                    } else {
                        split8(qg, hi, lo);
                        st16(sm, X_QG + chunk_mn(s0, ci, 1024, 1024), hi);
                        st16(sm, X_QG_LO + chunk_mn(s0, ci, 1024, 1024), lo);
                    }
                }
                float bw = (hf == 0) ? t1f : 1.f;  // e^{G_63 - G_t}: product over (t, 63]
#pragma unroll
                for (int c8 = 3; c8 >= 0; --c8) {
                    float kt[8];
#pragma unroll
                    for (int w = 7; w >= 0; --w) {
                        const int u = 8 * c8 + w, t = 32 * hf + u;
                        kt[w] = bf16_at(sm, RAW_K + t * 256 + ci * 2) * bw;
                        bw *= al[u];
                    }
                    const int s0 = 32 * hf + 8 * c8;
                    uint4 hi, lo;
                    split8(kt, hi, lo);
                    st16(sm, X_KT_HI + chunk_k(ci, s0, 128), hi);
                    st16(sm, X_KT_LO + chunk_k(ci, s0, 128), lo);
                }
            }
            fence_async_smem();
            fence_before();
            __syncthreads();
            fence_after();
            // ---- MMA 2: W^T = KG T_b^T, U~^T = V^T T_b^T
            if (tid == 0) {
                const uint32_t idk = idesc_bf16(128, 64, false, false, false);
                const uint32_t idv = idesc_bf16(128, 64, true, false, false);
#pragma unroll
                for (int pass = 0; pass < 3; ++pass) {
                    const uint32_t a = sb + (pass == 2 ? X_KG_LO : X_KG_HI);
                    const uint32_t b = sb + (pass == 1 ? OFF_TB_LO : OFF_TB_HI);
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        mma(tmem + TM_WT, desc_k(a, 128, s), desc_k(b, 64, s), idk, (pass | s) != 0);
                }
                commit(mbar);  // W^T only: U~^T (below) keeps running while W is extracted
#pragma unroll
                for (int pass = 0; pass < 2; ++pass) {
                    const uint32_t b = sb + (pass == 1 ? OFF_TB_LO : OFF_TB_HI);
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        mma(tmem + TM_UT, desc_mn(sb + OFF_V, 8192, 1024, s), desc_k(b, 64, s), idv,
                            (pass | s) != 0);
                }
            }
            // ---- state pass (overlaps MMA 2): S_j -> snapshot, bf16 hi/lo operand (over the raw
            //      tiles, all read by now), decay by e^{G_63}
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int col0 = colhalf * 64 + cc * 32;
                float v[32];
                ld32(tl + TM_S + col0, v);
                for (int m = 0; m < p.M; ++m) {
                    if (s_trk[m] != j) continue;
                    float* snap = p.track_state + (((size_t)n * p.M + m) * H + h) * (kD * kD) +
                                  (size_t)row * kD + col0;
#pragma unroll
                    for (int q4 = 0; q4 < 32; q4 += 4)
                        reinterpret_cast<float4*>(snap + q4)[0] =
                            make_float4(v[q4], v[q4 + 1], v[q4 + 2], v[q4 + 3]);
                }
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    uint4 hi, lo;
                    split8(v + 8 * c8, hi, lo);
                    st16(sm, OFF_ST_HI + chunk_k(row, col0 + 8 * c8, 128), hi);
                    st16(sm, OFF_ST_LO + chunk_k(row, col0 + 8 * c8, 128), lo);
                }
#pragma unroll
                for (int q = 0; q < 32; ++q) v[q] *= s_gam[col0 + q];
                st32(tl + TM_S + col0, v);
            }
            wait_st();
            const bool ok2 = mbar_wait(mbar, phase, kWaitLimit);
            phase ^= 1;
            fence_after();
            if (__syncthreads_or(!ok2)) {
                timed_out = true;
                break;
            }
            // ---- W^T (lanes i, columns t) -> W operand (B, MN-major [i][t]) hi/lo
            {
                float v[32];
                ld32(tl + TM_WT + colhalf * 32, v);
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    uint4 hi, lo;
                    split8(v + 8 * c8, hi, lo);
                    const int t = colhalf * 32 + 8 * c8;
                    st16(sm, X_W_HI + chunk_mn(t, row, 1024, 1024), hi);
                    st16(sm, X_W_LO + chunk_mn(t, row, 1024, 1024), lo);
                }
            }
            fence_async_smem();
            fence_before();
            __syncthreads();
            fence_after();
            // ---- MMA 3: O^T = S^T QG^T ; U^T = U~^T - S^T W^T (O first: one commit then frees the
            //      S operand, the V tile and the W / QG tiles)
            if (tid == 0) {
                const uint32_t idu = idesc_bf16(128, 64, false, true, true);
                const uint32_t ido = idesc_bf16(128, 64, false, true, false);
                // bf16 outputs: S_hi QG_hi; fp32 outputs: + S_lo QG_hi + S_hi QG_lo
#pragma unroll
                for (int pass = 0; pass < (kBf16Out ? 1 : 3); ++pass) {
                    const uint32_t a = sb + (pass == 1 ? OFF_ST_LO : OFF_ST_HI);
                    const uint32_t b = sb + (pass == 2 ? X_QG_LO : X_QG);
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        mma(tmem + TM_OT, desc_k(a, 128, s), desc_mn(b, 1024, 1024, s), ido,
                            (pass | s) != 0);
                }
#pragma unroll
                for (int pass = 0; pass < 3; ++pass) {
                    const uint32_t a = sb + (pass == 2 ? OFF_ST_LO : OFF_ST_HI);
                    const uint32_t b = sb + (pass == 1 ? X_W_LO : X_W_HI);
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        mma(tmem + TM_UT, desc_k(a, 128, s), desc_mn(b, 1024, 1024, s), idu, 1u);
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
            if (more) {
                // every reader of the S operand region and of the V tile has completed
                prefetch_qkg(j + 1);
                prefetch_v(j + 1);
                cp_async_commit();
            }
            // ---- U^T (lanes c, columns s) -> UT operand (A, K-major [c][s]) hi/lo
            {
                float v[32];
                ld32(tl + TM_UT + colhalf * 32, v);
#pragma unroll
                for (int c8 = 0; c8 < 4; ++c8) {
                    uint4 hi, lo;
                    split8(v + 8 * c8, hi, lo);
                    const int s0 = colhalf * 32 + 8 * c8;
                    st16(sm, X_UT_HI + chunk_k(row, s0, 128), hi);
                    st16(sm, X_UT_LO + chunk_k(row, s0, 128), lo);
                }
            }
            fence_async_smem();
            fence_before();
            __syncthreads();
            fence_after();
            // ---- MMA 4: O^T += U^T P^T ; S^T += U^T KT
            if (tid == 0) {
                const uint32_t ido = idesc_bf16(128, 64, false, false, false);
                const uint32_t ids = idesc_bf16(128, 128, false, false, false);
#pragma unroll
                for (int pass = 0; pass < (kBf16Out ? 1 : 3); ++pass) {
                    const uint32_t a = sb + (pass == 1 ? X_UT_LO : X_UT_HI);
                    const uint32_t b = sb + (pass == 2 ? OFF_P_LO : OFF_P);
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        mma(tmem + TM_OT, desc_k(a, 128, s), desc_k(b, 64, s), ido, 1u);
                }
                commit(mbar);  // the outputs; the state update below finishes in the background
#pragma unroll
                for (int pass = 0; pass < 3; ++pass) {
                    const uint32_t a = sb + (pass == 2 ? X_UT_LO : X_UT_HI);
                    const uint32_t b = sb + (pass == 1 ? X_KT_LO : X_KT_HI);
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        mma(tmem + TM_S, desc_k(a, 128, s), desc_k(b, 128, s), ids, 1u);
                }
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
                float v[32];
                ld32(tl + TM_OT + colhalf * 32, v);
                if constexpr (kBf16Out) {
                    // through shared memory (the T_b region, free now) for 16-byte row stores
                    __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(sm + OFF_TB_HI);
#pragma unroll
                    for (int q = 0; q < 32; ++q)
                        ob[(colhalf * 32 + q) * kD + row] = __float2bfloat16_rn(v[q]);
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
                    for (int q = 0; q < 32; ++q) {
                        const int t = colhalf * 32 + q;
                        if (t < Lc) store1<false>(p.out, ((size_t)(c0 + t) * H + h) * kD + row, v[q]);
                    }
                }
            }
        } else {
            // ---- fallback: this chunk token by token on CUDA cores (warps 0-3, a row each)
            float* alpha = reinterpret_cast<float*>(sm + X_ALPHA);
#pragma unroll
            for (int u = 0; u < 32; ++u) alpha[(32 * hf + u) * kD + ci] = al[u];
            fence_before();
            __syncthreads();
            fence_after();
            {
                // thread (row c, column half) keeps 64 state columns in registers; the two
                // half-row dot products meet in shared memory
                float* red = reinterpret_cast<float*>(sm + X_RED);  // [2 dots][2 halves][128]
                const int c = row;
                float sv[64];
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    float v[32];
                    ld32(tl + TM_S + colhalf * 64 + cc * 32, v);
#pragma unroll
                    for (int q = 0; q < 32; ++q) sv[cc * 32 + q] = v[q];
                }
                for (int m = 0; m < p.M; ++m) {
                    if (s_trk[m] != j) continue;
                    float* snap = p.track_state + (((size_t)n * p.M + m) * H + h) * (kD * kD) +
                                  (size_t)c * kD + colhalf * 64;
#pragma unroll
                    for (int q4 = 0; q4 < 64; q4 += 4)
                        reinterpret_cast<float4*>(snap + q4)[0] =
                            make_float4(sv[q4], sv[q4 + 1], sv[q4 + 2], sv[q4 + 3]);
                }
                for (int t = 0; t < Lc; ++t) {
                    float d1 = 0.f;
#pragma unroll
                    for (int q = 0; q < 64; ++q) {
                        const int i = colhalf * 64 + q;
                        sv[q] *= alpha[t * kD + i];
                        d1 = fmaf(sv[q], bf16_at(sm, RAW_K + t * 256 + i * 2), d1);
                    }
                    red[colhalf * 128 + c] = d1;
                    __syncthreads();
                    d1 = red[c] + red[128 + c];
                    const float vt = bf16_at(sm, OFF_V + chunk_mn(c & ~7, t, 8192, 1024) + (c & 7) * 2);
                    const float uu = s_beta[t] * (vt - d1);
                    float o = 0.f;
#pragma unroll
                    for (int q = 0; q < 64; ++q) {
                        const int i = colhalf * 64 + q;
                        sv[q] = fmaf(uu, bf16_at(sm, RAW_K + t * 256 + i * 2), sv[q]);
                        o = fmaf(sv[q], bf16_at(sm, RAW_Q + t * 256 + i * 2) * p.scale, o);
                    }
                    red[256 + colhalf * 128 + c] = o;
                    __syncthreads();
                    if (colhalf == 0)
                        store1<kBf16Out>(p.out, ((size_t)(c0 + t) * H + h) * kD + c,
                                         red[256 + c] + red[384 + c]);
                }
#pragma unroll
                for (int cc = 0; cc < 2; ++cc) {
                    float v[32];
#pragma unroll
                    for (int q = 0; q < 32; ++q) v[q] = sv[cc * 32 + q];
                    st32(tl + TM_S + colhalf * 64 + cc * 32, v);
                }
                wait_st();
            }
            fence_before();
            __syncthreads();
            fence_after();
            if (more) {
                prefetch_qkg(j + 1);
                prefetch_v(j + 1);
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
        // give in-flight MMAs a bounded chance to drain before TMEM is released
        mbar_wait(mbar, phase, kWaitLimit);
        if (pending_s) mbar_wait(mbar_s, phase_s, kWaitLimit);
    } else if (fin >= 0) {
        float* SD = p.pool + ((size_t)fin * H + h) * (kD * kD);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
            const int col0 = colhalf * 64 + cc * 32;
            float v[32];
            ld32(tl + TM_S + col0, v);
#pragma unroll
            for (int q4 = 0; q4 < 32; q4 += 4)
                reinterpret_cast<float4*>(SD + (size_t)row * kD + col0 + q4)[0] =
                    make_float4(v[q4], v[q4 + 1], v[q4 + 2], v[q4 + 3]);
        }
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

bool prefill_tc_supported(const PrefillArgs& p, bool bf16_in) { return bf16_in && p.M <= kTrackTc; }

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
