// verify.cu -- kda_spec_verify: speculative verify from one checkpoint per
// request, recording what the commit needs.
//
// vLLM PR 51855 page (RecoverSSM), implementation breakdown items 1 and 3:
// verify only reads the checkpoint, computes the output at each speculative
// position and writes the fp32 correction u and the activation-dtype key and
// raw gate into per-request record buffers of shape (heads, positions, d) and
// (heads, positions, 2 d).
//
// The K positions are evaluated in chunk form against the checkpoint S_0
// (G_t = sum_{u<=t} g_u per key channel):
//   u_t = beta_t (v_t - (k_t e^{G_t}) . S_0 - sum_{s<t} A_ts u_s),  A_ts = sum_i k_ti k_si e^{G_ti - G_si}
//   o_t = (q_t e^{G_t}) . S_0 + sum_{s<=t} P_ts u_s,                P_ts = sum_i q_ti k_si e^{G_ti - G_si}
// which is exactly K sequential steps of the recurrence.
//
// The work is a stream of 64 KiB checkpoints, one per (request, head) unit.
// Two persistent CTAs per SM (256 threads, ~100 KiB of shared memory and 256
// TMEM columns each) walk their units one after another; while one waits for
// its MMAs or its next checkpoint the other computes.  Per unit:
//   - the checkpoint arrives by TMA (a two-dimensional tensor map over the
//     pool, 128-byte swizzle, four [128 rows x 32 fp32] boxes, or two
//     [128 x 64] boxes for 16-bit states, widened exactly), requested as
//     soon as the previous unit's rows were converted; the token rows and raw
//     beta words arrive by cp.async one unit ahead;
//   - each thread converts 64 columns of one checkpoint row into bf16 hi + lo
//     in TMEM, the A operand (lane = value channel) of D = S_0^T [K_G; Q_G]^T
//     (M = 128, N = 2K padded to 16, K = 128): 16 MMAs, the hi / lo halves of
//     the gated keys and queries side by side along N;
//   - warps 0-3 write the gated keys / queries, warps 4-7 the K x K factors
//     (from mid-reference decay tables, one dot product per entry);
//   - after the MMAs, each of the 128 rows reads its 2K results from TMEM and
//     solves its K-step triangular system in registers.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "kda_common.cuh"
#include "kda_host.h"
#include "umma.cuh"

namespace kda {
namespace {

using namespace umma;

constexpr int kVThreads = 256;          // 8 warps: two per TMEM lane quarter
constexpr int kMaxVerifyK = 16;
constexpr int kMaxUnitsPerCta = 512;    // per-CTA unit table in shared memory
constexpr uint32_t kVWaitLimit = 1u << 18;  // polls of ~4 us (try_wait suspends): ~1 s; a checkpoint or an MMA batch lands in microseconds

struct VerifyArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* beta_raw;
    const void* gate_raw;
    int32_t K;
    const int32_t* q_len;
    int32_t H;
    float scale;
    uint32_t flags;
    int64_t P;
    const int32_t* ckpt;
    float* rec_u;
    void* rec_kg;
    void* out;
    int32_t* dev_status;
    int32_t n_units;
    int32_t st;  // StateType of the pool
};

constexpr uint32_t align16(uint32_t x) { return (x + 15u) & ~15u; }

// Shared-memory plan for a compile-time bound KC on K and the activation element size ES.
// Every region starts on a 16-byte boundary (cp.async and vector accesses).
template <int KC, int ES>
struct VLayout {
    static constexpr int NB = 2 * KC < 16 ? 16 : 2 * KC;  // MMA N of one hi or lo half
    static constexpr int TLD = 132;                        // pair-table row stride (floats)
    static constexpr uint32_t RAW = 0;                     // 64 KiB checkpoint (TMA, swizzled)
    static constexpr uint32_t BT = 65536;                  // [B_hi; B_lo] tile, K-major
    static constexpr uint32_t BT_BYTES = 2 * NB * 256;
    static constexpr uint32_t KQG = BT + BT_BYTES;         // k, q, g rows [3][KC][128]
    static constexpr uint32_t KQG_BYTES = 3 * KC * 128 * ES;
    static constexpr uint32_t VB = align16(KQG + KQG_BYTES);  // 2 x v rows [KC][128]
    static constexpr uint32_t VB_BYTES = KC * 128 * ES;
    static constexpr uint32_t AP = align16(VB + 2 * VB_BYTES);   // [KC][KC] fp32
    static constexpr uint32_t RED = align16(AP + KC * KC * 4);   // [4 warps][KC][KC]
    static constexpr uint32_t BETA = align16(RED + 4 * KC * KC * 4);  // [KC] activated beta
    static constexpr uint32_t BRAW = align16(BETA + KC * 4);     // [KC] 4-byte words holding raw beta
    static constexpr uint32_t NRM = align16(BRAW + KC * 4);      // [2][KC] L2 factors of k, q
    static constexpr uint32_t TAB = align16(NRM + 2 * KC * 4);   // [3][KC][TLD] fp32 (K <= 8)
    static constexpr uint32_t TAB_BYTES = KC <= 8 ? 3 * KC * TLD * 4 : 0;
    static constexpr uint32_t META = align16(TAB + TAB_BYTES);   // [kMaxUnitsPerCta] (slot, q_len)
    static constexpr uint32_t MBAR = META + kMaxUnitsPerCta * 8; // checkpoint, MMA
    static constexpr uint32_t END = MBAR + 2 * 8 + 16;
    static constexpr size_t SMEM = END + 1024;  // + alignment slack
    static_assert(BT % 1024 == 0 && BT_BYTES % 1024 == 0, "swizzled tiles on 1 KiB boundaries");
    static_assert(KQG % 16 == 0 && VB % 16 == 0 && TAB % 16 == 0 && META % 8 == 0, "region alignment");
    static_assert(SMEM <= 232448, "verify shared memory plan exceeds the per-CTA limit");
};

// TMEM columns: checkpoint operand [S hi (64) | S lo (64)], then the accumulator [D_hi | D_lo]
constexpr uint32_t TV_SA = 0, TV_D = 128, TV_COLS = 256;

constexpr float kVFactorMax = 1.8446744e19f;  // 2^64: largest decay factor the pair tables carry

template <bool kBf16>
__device__ __forceinline__ float act_at(const uint8_t* p, int idx) {
    if constexpr (kBf16)
        return __uint_as_float((uint32_t)(reinterpret_cast<const uint16_t*>(p)[idx]) << 16);
    else
        return reinterpret_cast<const float*>(p)[idx];
}

template <int KC, bool kBf16In, bool kBf16Out>
__global__ void __launch_bounds__(kVThreads, 2)
    verify_kernel(const __grid_constant__ CUtensorMap tmap, const VerifyArgs a) {
    constexpr int ES = kBf16In ? 2 : 4;
    using Lay = VLayout<KC, ES>;
    constexpr int NB = Lay::NB;
    constexpr int CPR = 128 * ES / 16;  // 16-byte chunks per token row
    static_assert(TV_D + 2 * NB <= TV_COLS, "TMEM plan");

    extern __shared__ uint8_t vraw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(vraw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(sm);
    const uint32_t sb4 = sb >> 4;
    int2* meta = reinterpret_cast<int2*>(sm + Lay::META);
    uint64_t* mbars = reinterpret_cast<uint64_t*>(sm + Lay::MBAR);  // checkpoint, MMA
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(mbars + 2);
    float* sbeta = reinterpret_cast<float*>(sm + Lay::BETA);
    float* ap = reinterpret_cast<float*>(sm + Lay::AP);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3, colhalf = warp >> 2;
    const int row = quarter * 32 + lane;
    const int i = tid & 127;  // channel passes: key channel
    const int H = a.H, K = a.K;
    const int G = gridDim.x;
    const int nu = (a.n_units - (int)blockIdx.x + G - 1) / G;  // units of this CTA

    // ---- unit table: checkpoint slot and accepted length (0 = skipped)
    for (int idx = tid; idx < nu; idx += kVThreads) {
        const int unit = blockIdx.x + idx * G;
        const int r = unit / H, h = unit - r * H;
        const int slot = a.ckpt[r];
        int ql = a.q_len ? a.q_len[r] : K;
        const bool slot_ok = slot >= 0 && slot < a.P;
        const bool len_ok = ql >= 0 && ql <= K;
        if (h == 0) {
            if (slot >= a.P) report(a.dev_status, KDA_DEV_BAD_SLOT);
            if (!len_ok) report(a.dev_status, KDA_DEV_BAD_ACCEPT);
        }
        if (!(slot_ok && len_ok)) ql = 0;
        meta[idx] = make_int2(slot, ql);
    }
    if (warp == 0) tmem_alloc(smem_u32(s_tmem), TV_COLS);
    if (tid == 0) {
        mbar_init(smem_u32(mbars), 1);
        mbar_init(smem_u32(mbars + 1), 1);
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);

    auto unit_rh = [&](int idx, int& r, int& h) {
        const int unit = blockIdx.x + idx * G;
        r = unit / H;
        h = unit - r * H;
    };
    // checkpoint of unit idx (q_len > 0) -> RAW, completing on the checkpoint barrier (one thread)
    auto request_ckpt = [&](int idx) {
        int r, h;
        unit_rh(idx, r, h);
        const uint32_t mb = smem_u32(mbars);
        const int y = (meta[idx].x * H + h) * 128;
        if (a.st == kStateF32) {  // four [128 x 32] fp32 boxes
            mbar_expect_tx(mb, 65536u);
#pragma unroll
            for (int p = 0; p < 4; ++p) tma_load_2d(sb + Lay::RAW + p * 16384, &tmap, 32 * p, y, mb);
        } else {  // two [128 x 64] 16-bit boxes
            mbar_expect_tx(mb, 32768u);
#pragma unroll
            for (int p = 0; p < 2; ++p) tma_load_2d(sb + Lay::RAW + p * 16384, &tmap, 64 * p, y, mb);
        }
    };
    // token rows of unit idx: k, q, g -> KQG, v -> VB[idx & 1], raw beta words -> BRAW;
    // rows past the accepted length are zero-filled
    auto prefetch_tokens = [&](int idx) {
        const int ql = meta[idx].y;
        int r, h;
        unit_rh(idx, r, h);
        for (int e2 = tid; e2 < 4 * KC * CPR; e2 += kVThreads) {
            const int x = e2 / (KC * CPR), rem = e2 - x * KC * CPR, t = rem / CPR, ch = rem - t * CPR;
            const void* src = x == 0 ? a.k : x == 1 ? a.q : x == 2 ? a.gate_raw : a.v;
            const bool ok = t < ql;
            const size_t e = ok ? (((size_t)r * K + t) * H + h) * 128 : 0;
            const uint32_t dst = x < 3 ? Lay::KQG + (uint32_t)((x * KC + t) * 128 * ES + ch * 16)
                                       : Lay::VB + (uint32_t)(idx & 1) * Lay::VB_BYTES +
                                             (uint32_t)(t * 128 * ES + ch * 16);
            cp_async16(sb + dst, static_cast<const uint8_t*>(src) + e * ES + (ok ? ch * 16 : 0),
                       ok ? 16u : 0u);
        }
        if (tid < KC) {  // the aligned 4-byte word holding beta of position tid
            const bool ok = tid < ql;
            const size_t e = ok ? ((size_t)r * K + tid) * H + h : 0;
            cp_async4(sb + Lay::BRAW + (uint32_t)tid * 4,
                      static_cast<const uint8_t*>(a.beta_raw) + ((e * ES) & ~(size_t)3), ok ? 4u : 0u);
        }
    };
    // checkpoint rows, column quarter cq_ (32 columns of row `row`) -> TMEM operand (hi | lo)
    auto convert = [&](int cq_) {
        float x[32];
        if (a.st == kStateF32) {
            // box cq_ holds columns 32 cq_ .. +31: eight 16-byte pieces per 128-byte row
            const uint8_t* raw = sm + Lay::RAW + (uint32_t)cq_ * 16384u;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                const float4 f = *reinterpret_cast<const float4*>(raw + row * 128 + ((m ^ (row & 7)) << 4));
                x[4 * m] = f.x;
                x[4 * m + 1] = f.y;
                x[4 * m + 2] = f.z;
                x[4 * m + 3] = f.w;
            }
        } else {
            // box cq_ / 2 holds columns 64 (cq_ / 2) .. +63; this quarter is pieces 4 (cq_ & 1) .. +3
            const uint8_t* raw = sm + Lay::RAW + (uint32_t)(cq_ >> 1) * 16384u;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int piece = 4 * (cq_ & 1) + m;
                const uint4 w = *reinterpret_cast<const uint4*>(raw + row * 128 + ((piece ^ (row & 7)) << 4));
                const float4 lo = a.st == kStateBF16 ? State<kStateBF16>::widen(make_uint2(w.x, w.y))
                                                     : State<kStateF16>::widen(make_uint2(w.x, w.y));
                const float4 hi = a.st == kStateBF16 ? State<kStateBF16>::widen(make_uint2(w.z, w.w))
                                                     : State<kStateF16>::widen(make_uint2(w.z, w.w));
                x[8 * m] = lo.x;
                x[8 * m + 1] = lo.y;
                x[8 * m + 2] = lo.z;
                x[8 * m + 3] = lo.w;
                x[8 * m + 4] = hi.x;
                x[8 * m + 5] = hi.y;
                x[8 * m + 6] = hi.z;
                x[8 * m + 7] = hi.w;
            }
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            uint32_t sh[8], sl[8];
#pragma unroll
            for (int q2 = 0; q2 < 8; ++q2) split2(x[16 * hh + 2 * q2], x[16 * hh + 2 * q2 + 1], sh[q2], sl[q2]);
            const uint32_t col = TV_SA + (uint32_t)cq_ * 16u + 8u * hh;
            st8u(tl + col, sh);
            st8u(tl + col + 64, sl);
        }
    };

    // ---- prologue: the first unit's checkpoint and token rows
    uint32_t ph_raw = 0, ph_mma = 0;
    bool raw_pend = false, mma_pend = false;
    if (nu > 0) {
        if (meta[0].y > 0) {
            if (tid == 0) request_ckpt(0);
            raw_pend = true;
        }
        prefetch_tokens(0);
        cp_async_commit();
    }
    bool timed_out = false;

    for (int it = 0; it < nu; ++it) {
        const int ql = meta[it].y;
        int r, h;
        unit_rh(it, r, h);
        // ---- this unit's token rows (its checkpoint is waited for after the channel work below,
        //      which does not read it)
        cp_async_wait_all();
        __syncthreads();
        if (tid < KC) {
            float bv = 0.f;
            if (tid < ql) {
                const uint32_t w = reinterpret_cast<const uint32_t*>(sm + Lay::BRAW)[tid];
                const size_t e = ((size_t)r * K + tid) * H + h;
                bv = beta_act(kBf16In ? __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16))
                                      : __uint_as_float(w),
                              a.flags);
            }
            sbeta[tid] = bv;
        }
        // ---- KDA_QK_L2NORM: the factors of the key and query rows (a warp per row)
        float* nrm = reinterpret_cast<float*>(sm + Lay::NRM);
        const bool l2 = (a.flags & KDA_QK_L2NORM) != 0;
        if (l2) {
            const uint8_t* kqg = sm + Lay::KQG;
            for (int t = warp; t < KC; t += kVThreads / 32) {
                float sk = 0.f, sq = 0.f;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float kx = act_at<kBf16In>(kqg, t * 128 + 4 * lane + e);
                    const float qx = act_at<kBf16In>(kqg, (KC + t) * 128 + 4 * lane + e);
                    sk = fmaf(kx, kx, sk);
                    sq = fmaf(qx, qx, sq);
                }
                warp_sum2(sk, sq);
                if (lane == 0) {
                    nrm[t] = l2norm_factor(sk);
                    nrm[KC + t] = l2norm_factor(sq);
                }
            }
        }
        if (l2) __syncthreads();  // the factors above, for every channel thread below
        // ---- channel i: gates; warps 0-3 the gated keys / queries and the key / raw gate
        //      records, warps 4-7 the K x K factors
        {
            const uint8_t* kqg = sm + Lay::KQG;
            float kt[KC], qt[KC], at[KC], iv[KC];  // key, scaled query, alpha, 1 / alpha
            with_gate_form(a.flags, [&](uint32_t form) {
#pragma unroll
                for (int t = 0; t < KC; ++t) {
                    kt[t] = act_at<kBf16In>(kqg, t * 128 + i);
                    qt[t] = act_at<kBf16In>(kqg, (KC + t) * 128 + i) * a.scale;
                    if (l2) {
                        kt[t] *= nrm[t];
                        qt[t] *= nrm[KC + t];
                    }
                    // rows past the accepted length arrived zero-filled: finite, then replaced
                    const Decay dc = decay_of(act_at<kBf16In>(kqg, (2 * KC + t) * 128 + i), form);
                    at[t] = t < ql ? dc.a : 1.f;
                    iv[t] = t < ql ? dc.inv : 1.f;
                }
            });
            if (warp < 4) {
                uint16_t* bt = reinterpret_cast<uint16_t*>(sm + Lay::BT);
                auto put = [&](int n, float val) {
                    const __nv_bfloat16 hi = __float2bfloat16_rn(val);
                    const __nv_bfloat16 lo = __float2bfloat16_rn(val - __bfloat162float(hi));
                    bt[(chunk_k(n, i & ~7, 2 * NB) + (i & 7) * 2) >> 1] = __bfloat16_as_ushort(hi);
                    bt[(chunk_k(NB + n, i & ~7, 2 * NB) + (i & 7) * 2) >> 1] = __bfloat16_as_ushort(lo);
                };
                float cum = 1.f;  // e^{G_t}
#pragma unroll
                for (int t = 0; t < KC; ++t) {
                    cum *= at[t];
                    put(t, kt[t] * cum);
                    put(KC + t, qt[t] * cum);
                }
#pragma unroll
                for (int n = 2 * KC; n < NB; ++n) put(n, 0.f);
                // records: key and raw gate exactly as given, zeros past the accepted length
                const size_t rec0 = ((size_t)r * H + h) * K;
                for (int e = tid; e < 2 * K * CPR; e += 128) {
                    const int t = e / (2 * CPR), rem = e - t * 2 * CPR, half = rem / CPR, ch = rem - half * CPR;
                    uint4 val = make_uint4(0u, 0u, 0u, 0u);
                    if (t < ql)
                        val = *reinterpret_cast<const uint4*>(
                            sm + Lay::KQG + (uint32_t)(((half ? 2 * KC : 0) + t) * 128 * ES + ch * 16));
                    *reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.rec_kg) +
                                              ((rec0 + t) * 2 * 128 + half * 128) * ES + ch * 16) = val;
                }
            } else {
                const int wg = warp - 4;
                bool fallback = true;
                if constexpr (KC <= 8) {
                    // Tables with the reference at position m = KC/2 (factors span at most KC/2
                    // steps): L_k[t] = k_t e^{G_t - G_m}, L_q[t] = q_t e^{G_t - G_m},
                    // R[s] = k_s e^{G_m - G_s}; then A_ts = L_k[t] . R[s], P_ts = L_q[t] . R[s].
                    constexpr int MID = KC / 2, TLD = Lay::TLD;
                    float* lk = reinterpret_cast<float*>(sm + Lay::TAB);
                    float* lq = lk + KC * TLD;
                    float* rk = lq + KC * TLD;
                    lk[MID * TLD + i] = kt[MID];
                    lq[MID * TLD + i] = qt[MID];
                    rk[MID * TLD + i] = kt[MID];
                    float e = 1.f, rf = 1.f;
#pragma unroll
                    for (int t = MID + 1; t < KC; ++t) {
                        e *= at[t];
                        rf *= iv[t];
                        lk[t * TLD + i] = kt[t] * e;
                        lq[t * TLD + i] = qt[t] * e;
                        rk[t * TLD + i] = kt[t] * rf;
                    }
                    float big = rf;
                    e = rf = 1.f;
#pragma unroll
                    for (int t = MID - 1; t >= 0; --t) {
                        e *= iv[t + 1];
                        rf *= at[t + 1];
                        lk[t * TLD + i] = kt[t] * e;
                        lq[t * TLD + i] = qt[t] * e;
                        rk[t * TLD + i] = kt[t] * rf;
                    }
                    big = fmaxf(big, e);
                    fallback = bar_named_or(1, 128, !(big <= kVFactorMax));
                    if (!fallback) {
                        // entry [x0][x1]: P (query x1, key x0) if x0 <= x1, else A (x0, x1); two
                        // threads per entry, 64 channels each
                        constexpr int NIT = KC * KC * 2;
                        constexpr unsigned MASK = NIT >= 32 ? 0xffffffffu : (1u << NIT) - 1u;
                        for (int e2 = i; e2 < NIT; e2 += 128) {
                            const int entry = e2 >> 1, half = e2 & 1;
                            const int x0 = entry / KC, x1 = entry - x0 * KC;
                            const float* lrow = (x0 <= x1 ? lq + x1 * TLD : lk + x0 * TLD) + 64 * half;
                            const float* rrow = rk + (x0 <= x1 ? x0 : x1) * TLD + 64 * half;
                            float acc = 0.f;
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const float4 l4 = *reinterpret_cast<const float4*>(lrow + 4 * j);
                                const float4 r4 = *reinterpret_cast<const float4*>(rrow + 4 * j);
                                acc = fmaf(l4.x, r4.x, acc);
                                acc = fmaf(l4.y, r4.y, acc);
                                acc = fmaf(l4.z, r4.z, acc);
                                acc = fmaf(l4.w, r4.w, acc);
                            }
                            acc += __shfl_xor_sync(MASK, acc, 1);
                            if (half == 0) ap[entry] = acc;
                        }
                    }
                }
                if (fallback) {
                    // pair sums over channels, e^{G_t - G_s} as running products of alpha:
                    // value [x0][x1] = P (x0 <= x1) or A (x0 > x1), summed over the warp's channels
                    float(*red)[KC][KC] = reinterpret_cast<float(*)[KC][KC]>(sm + Lay::RED);
                    if constexpr (KC <= 8) {
                        constexpr int NV = KC * KC < 32 ? 32 : KC * KC;
                        float vals[NV];
#pragma unroll
                        for (int e = 0; e < NV; ++e) vals[e] = 0.f;
#pragma unroll
                        for (int s0 = 0; s0 < KC; ++s0) {
                            float dec = 1.f;
#pragma unroll
                            for (int t = s0; t < KC; ++t) {
                                if (t > s0) dec *= at[t];
                                const bool live = t < ql;
                                vals[s0 * KC + t] = live ? qt[t] * kt[s0] * dec : 0.f;
                                if (t > s0) vals[t * KC + s0] = live ? kt[t] * kt[s0] * dec : 0.f;
                            }
                        }
                        // butterfly reduce-scatter: lane l ends with the totals of entries l*M .. l*M+M-1
                        int nn = NV;
#pragma unroll
                        for (int off = 16; off >= 1; off >>= 1) {
                            const bool upper = (lane & off) != 0;
                            const int half = nn / 2;
#pragma unroll
                            for (int e = 0; e < NV / 2; ++e) {
                                if (e < half) {
                                    const float send = upper ? vals[e] : vals[e + half];
                                    const float keep = upper ? vals[e + half] : vals[e];
                                    vals[e] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                                }
                            }
                            nn = half;
                        }
                        constexpr int M = NV / 32;
#pragma unroll
                        for (int e = 0; e < M; ++e) {
                            const int idx = lane * M + e;
                            if (idx < KC * KC) red[wg][idx / KC][idx % KC] = vals[e];
                        }
                    } else {
#pragma unroll
                        for (int s0 = 0; s0 < KC; ++s0) {
                            float dec = 1.f;
#pragma unroll
                            for (int t = s0; t < KC; ++t) {
                                if (t > s0) dec *= at[t];
                                const bool live = t < ql;
                                const float pp = warp_sum(live ? qt[t] * kt[s0] * dec : 0.f);
                                if (lane == 0) red[wg][s0][t] = pp;
                                if (t > s0) {
                                    const float pa = warp_sum(live ? kt[t] * kt[s0] * dec : 0.f);
                                    if (lane == 0) red[wg][t][s0] = pa;
                                }
                            }
                        }
                    }
                    bar_named(1, 128);  // warps 4-7
                    for (int e = i; e < KC * KC; e += 128) {
                        const int x0 = e / KC, x1 = e - x0 * KC;
                        ap[e] = (red[0][x0][x1] + red[1][x0][x1]) + (red[2][x0][x1] + red[3][x0][x1]);
                    }
                }
            }
        }
        // ---- this unit's checkpoint (every thread waits on its barrier) -> TMEM operand (all
        //      warps, 64 columns each).  A bf16 checkpoint is used where it landed: the two
        //      64-channel boxes of 128 rows, 128-byte swizzled, are the K-major shared-memory
        //      A operand of the MMA (its hi part, lo = 0), so it needs no conversion; it then
        //      holds the staging buffer until the MMA has read it.
        const bool a_in_smem = a.st == kStateBF16;
        if (raw_pend) {
            if (!mbar_wait(smem_u32(mbars), ph_raw, kVWaitLimit)) timed_out = true;
            ph_raw ^= 1u;
            raw_pend = false;
        }
        if (ql > 0 && !timed_out && !a_in_smem) {
            convert(2 * colhalf);
            convert(2 * colhalf + 1);
            wait_st();
        }
        fence_async_smem();
        fence_before();
        if (__syncthreads_or(timed_out)) {
            timed_out = true;
            break;
        }
        fence_after();
        // ---- the next unit's checkpoint (RAW has been converted; requested by warp 1, so that
        //      thread 0 goes straight to the MMAs; for a bf16 checkpoint after the MMAs have read
        //      it, below) and token rows, then this unit's MMAs:
        //      D = S_hi [B_hi; B_lo]^T + S_lo B_hi^T
        const bool next_ckpt = it + 1 < nu && meta[it + 1].y > 0;
        if (next_ckpt && !a_in_smem) {
            if (tid == 32) request_ckpt(it + 1);
            raw_pend = true;
        }
        if (ql > 0) {
            if (tid == 0) {
                const uint32_t id2 = idesc_bf16(128, 2 * NB, false, false, false);
                const uint32_t id1 = idesc_bf16(128, NB, false, false, false);
                const uint32_t b4 = sb4 + Lay::BT / 16;
                if (a_in_smem) {
                    // a bf16 checkpoint splits exactly into hi with lo = 0: its lo products are zero
                    const uint32_t a4 = sb4 + Lay::RAW / 16;
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        mma(tmem + TV_D, desc_k4(a4, 128, s), desc_k4(b4, 2 * NB, s), id2, s != 0);
                } else {
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        mma_ta(tmem + TV_D, tmem + TV_SA + 8 * s, desc_k4(b4, 2 * NB, s), id2, s != 0);
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        mma_ta(tmem + TV_D, tmem + TV_SA + 64 + 8 * s, desc_k4(b4, 2 * NB, s), id1, 1u);
                }
                commit(smem_u32(mbars + 1));
            }
            mma_pend = true;
        }
        // v rows of this unit stay in VB[it & 1] for the solve; the next unit's go to the other
        if (it + 1 < nu) prefetch_tokens(it + 1);
        cp_async_commit();
        if (mma_pend) {
            if (tid == 0 && !mbar_wait(smem_u32(mbars + 1), ph_mma, kVWaitLimit)) timed_out = true;
            ph_mma ^= 1u;
            mma_pend = false;
        }
        fence_before();
        if (__syncthreads_or(timed_out)) {
            timed_out = true;
            break;
        }
        fence_after();
        // a bf16 checkpoint: the MMAs have read it, so the next one may land in its place
        if (next_ckpt && a_in_smem) {
            if (tid == 32) request_ckpt(it + 1);
            raw_pend = true;
        }
        // ---- rows (warps 0-3): triangular solve, outputs, u records
        if (warp < 4) {
            const size_t rec0 = ((size_t)r * H + h) * K;
            const int c = tid;
            float d[2 * NB];
            if (ql > 0) {
#pragma unroll
                for (int q16 = 0; q16 < 2 * NB / 16; ++q16) {
                    float v16[16];
                    ld16(tl + TV_D + 16 * q16, v16);
#pragma unroll
                    for (int e = 0; e < 16; ++e) d[16 * q16 + e] = v16[e];
                }
            }
            const uint8_t* vb = sm + Lay::VB + (uint32_t)(it & 1) * Lay::VB_BYTES;
            float u[KC];
#pragma unroll
            for (int t = 0; t < KC; ++t) {
                u[t] = 0.f;
                if (t >= K) continue;
                const size_t th = ((size_t)r * K + t) * H + h;
                float o = 0.f;
                if (t < ql) {
                    float acc = d[t] + d[NB + t];
#pragma unroll
                    for (int s0 = 0; s0 < t; ++s0) acc = fmaf(ap[t * KC + s0], u[s0], acc);
                    u[t] = sbeta[t] * (act_at<kBf16In>(vb, t * 128 + c) - acc);
                    o = d[KC + t] + d[NB + KC + t];
#pragma unroll
                    for (int s0 = 0; s0 <= t; ++s0) o = fmaf(ap[s0 * KC + t], u[s0], o);
                }
                store1<kBf16Out>(a.out, th * kD + c, o);
                a.rec_u[(rec0 + t) * kD + c] = u[t];
            }
            fence_before();
        }
    }
    cp_async_wait_all();
    timed_out = __syncthreads_or(timed_out);
    if (timed_out) {
        if (tid == 0) {
            report(a.dev_status, KDA_DEV_TIMEOUT);
            // bounded drain of what may still be in flight before shared memory and TMEM are
            // released: the last checkpoint and MMA phases waited on (either may be the one that
            // timed out; a wait on a completed phase returns at once) and whatever was issued but
            // not yet waited on
            mbar_wait(smem_u32(mbars), ph_raw ^ 1u, kVWaitLimit);
            if (raw_pend) mbar_wait(smem_u32(mbars), ph_raw, kVWaitLimit);
            mbar_wait(smem_u32(mbars + 1), ph_mma ^ 1u, kVWaitLimit);
            if (mma_pend) mbar_wait(smem_u32(mbars + 1), ph_mma, kVWaitLimit);
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0) tmem_dealloc(tmem, TV_COLS);
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

template <int KC, bool I, bool O>
kda_status launch_kc(const CUtensorMap& map, const VerifyArgs& a, cudaStream_t s) {
    constexpr size_t smem = VLayout<KC, I ? 2 : 4>::SMEM;
    const int nsm = sm_count();
    if (nsm <= 0) return KDA_ERR_CUDA;
    cudaFuncSetAttribute(verify_kernel<KC, I, O>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    // all of the unified L1 / shared storage as shared memory, so two CTAs fit on an SM
    cudaFuncSetAttribute(verify_kernel<KC, I, O>, cudaFuncAttributePreferredSharedMemoryCarveout,
                         (int)cudaSharedmemCarveoutMaxShared);
    // two CTAs per SM when two shared-memory plans (plus the 1 KiB each CTA reserves) fit in an
    // SM's 228 KiB; registers allow two by the launch bounds, TMEM by 2 x 256 columns
    const int per_sm = 2 * (smem + 1024) <= 233472 ? 2 : 1;
    int grid = nsm * per_sm;
    if (grid > a.n_units) grid = a.n_units;
    const int need = (a.n_units + kMaxUnitsPerCta - 1) / kMaxUnitsPerCta;
    if (grid < need) grid = need;
    verify_kernel<KC, I, O><<<(unsigned)grid, kVThreads, smem, s>>>(map, a);
    return launch_status();
}

template <bool I, bool O>
kda_status launch(const CUtensorMap& map, const VerifyArgs& a, cudaStream_t s) {
    if (a.K <= 2) return launch_kc<2, I, O>(map, a, s);
    if (a.K <= 4) return launch_kc<4, I, O>(map, a, s);
    if (a.K <= 8) return launch_kc<8, I, O>(map, a, s);
    return launch_kc<16, I, O>(map, a, s);
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" kda_status kda_spec_verify(const void* q, const void* k, const void* v,
                                      const void* beta_raw, const void* gate_raw,
                                      kda_dtype in_dtype, int32_t R, int32_t K,
                                      const int32_t* q_len, int32_t H, int32_t dk, int32_t dv,
                                      float scale, uint32_t flags, const void* state_pool,
                                      int64_t P, const int32_t* ckpt_slot, float* rec_u,
                                      void* rec_kg, void* out, kda_dtype out_dtype,
                                      int32_t* dev_status, void* stream) {
    KDA_REQUIRE(R >= 0 && K >= 0 && H > 0 && P >= 0, KDA_ERR_INVALID_ARG);
    KDA_REQUIRE(dk == kD && dv == kD, KDA_ERR_UNSUPPORTED);
    KDA_REQUIRE(dtype_ok(in_dtype) && dtype_ok(out_dtype), KDA_ERR_UNSUPPORTED);
    KDA_REQUIRE(K <= kMaxVerifyK, KDA_ERR_UNSUPPORTED);
    KDA_REQUIRE(state_flags_ok(flags), KDA_ERR_UNSUPPORTED);
    if (R == 0 || K == 0) return KDA_OK;
    KDA_REQUIRE((int64_t)R * H < (1ll << 31), KDA_ERR_UNSUPPORTED);
    // the pool is read as a 2-D tensor of P*H*128 rows of 128 states (a TMA row coordinate each)
    KDA_REQUIRE(P * H * 128 < (1ll << 31), KDA_ERR_UNSUPPORTED);
    const void* ptrs[] = {q, k, v, beta_raw, gate_raw, state_pool, ckpt_slot, rec_u, rec_kg, out};
    for (const void* p : ptrs) KDA_REQUIRE(p != nullptr && aligned16(p), KDA_ERR_INVALID_ARG);
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return KDA_ERR_CUDA;
    CUtensorMap map;
    const int st = state_type(flags);
    const cuuint64_t rows = P > 0 ? (cuuint64_t)P * H * 128 : 128;
    const cuuint64_t dims[2] = {128, rows};
    // one 128-byte swizzle row per box row: 32 fp32 or 64 16-bit states
    const cuuint64_t strides[1] = {128 * (cuuint64_t)state_bytes(st)};
    const cuuint32_t box[2] = {st == kStateF32 ? 32u : 64u, 128};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType et = st == kStateF32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : st == kStateBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (enc(&map, et, 2, const_cast<void*>(state_pool), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return KDA_ERR_CUDA;
    const VerifyArgs a{q, k, v, beta_raw, gate_raw, K, q_len, H, scale, flags, P, ckpt_slot,
                       rec_u, rec_kg, out, dev_status, R * H, st};
    cudaStream_t s = as_stream(stream);
    const bool ib = in_dtype == KDA_BF16, ob = out_dtype == KDA_BF16;
    if (ib && ob) return launch<true, true>(map, a, s);
    if (ib) return launch<true, false>(map, a, s);
    if (ob) return launch<false, true>(map, a, s);
    return launch<false, false>(map, a, s);
}
