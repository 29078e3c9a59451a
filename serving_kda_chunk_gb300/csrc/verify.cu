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
// which is exactly K sequential steps of the recurrence.  One CTA per
// (request, head), 128 threads.  The 2K dot products of every state row with
// the gated keys and queries form one K S tile, D = S_0^T [K_G; Q_G]^T
// (M = 128 value channels, N = 2K padded to 16, K = 128 key channels), run on
// tcgen05 with the fp32 checkpoint split into bf16 hi + lo operands (three
// passes, fp32 accumulation in TMEM).  The checkpoint is read once with
// coalesced streaming loads straight into the swizzled operand tiles; the K x K
// factors A and P are built from running products of alpha; each thread then
// reads its row's 2K results from TMEM and solves the row's triangular system
// in registers.  Loops are specialised on a compile-time bound of K.
#include "kda_common.cuh"
#include "kda_host.h"
#include "umma.cuh"

namespace kda {
namespace {

constexpr int kVThreads = 256;  // 128 rows / channels; the upper half helps stage the checkpoint
constexpr int kMaxVerifyK = 16;

using namespace umma;

constexpr uint32_t kVWaitLimit = 1u << 22;  // polls; the MMA chain completes in microseconds

// KC: compile-time bound on K (2, 4, 8 or 16); NB = MMA N (K_G rows then Q_G rows).
template <int KC, bool kBf16In, bool kBf16Out>
__global__ void __launch_bounds__(kVThreads) verify_kernel(
    const void* __restrict__ q, const void* __restrict__ k, const void* __restrict__ v,
    const void* __restrict__ beta_raw, const void* __restrict__ gate_raw, int32_t K,
    const int32_t* __restrict__ q_len, int32_t H, float scale, uint32_t flags,
    const float* __restrict__ pool, int64_t P, const int32_t* __restrict__ ckpt,
    float* __restrict__ rec_u, void* __restrict__ rec_kg, void* __restrict__ out,
    int32_t* __restrict__ dev_status) {
    using A = Act<kBf16In>;
    constexpr int NB = 2 * KC < 16 ? 16 : 2 * KC;
    constexpr uint32_t ST_HI = 0, ST_LO = 32768, KQ_HI = 65536, KQ_LO = 65536 + NB * 256;
    constexpr uint32_t MISC = KQ_LO + NB * 256;
    extern __shared__ uint8_t vraw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(vraw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(sm);
    float(*AP)[KC] = reinterpret_cast<float(*)[KC]>(sm + MISC);               // A at [t][s], P at [s][t]
    float(*red)[KC][KC] = reinterpret_cast<float(*)[KC][KC]>(sm + MISC + KC * KC * 4);
    float* sbeta = reinterpret_cast<float*>(sm + MISC + 5 * KC * KC * 4);
    uint64_t* mbar = reinterpret_cast<uint64_t*>(sm + MISC + 5 * KC * KC * 4 + KC * 4 + 8 -
                                                 ((5 * KC * KC * 4 + KC * 4) & 7));
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(mbar + 1);

    const int unit = blockIdx.x;
    const int r = unit / H, h = unit - r * H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slot = ckpt[r];
    int ql = q_len ? q_len[r] : K;
    const bool slot_ok = slot >= 0 && slot < P;
    const bool len_ok = ql >= 0 && ql <= K;
    if (!(slot_ok && len_ok)) {
        if (tid == 0 && h == 0) {
            if (slot >= P) report(dev_status, KDA_DEV_BAD_SLOT);
            if (!len_ok) report(dev_status, KDA_DEV_BAD_ACCEPT);
        }
        ql = 0;
    }
    const size_t rec0 = ((size_t)r * H + h) * K;
    if (ql == 0) {
        if (tid < kD) {
            for (int t = 0; t < K; ++t) {
                const size_t th = ((size_t)r * K + t) * H + h;
                store1<kBf16Out>(out, th * kD + tid, 0.f);
                rec_u[(rec0 + t) * kD + tid] = 0.f;
                if (tid < 64) A::zero4(rec_kg, (rec0 + t) * 2 * kD + 4 * tid);
            }
        }
        return;
    }
    // ---- every load of this unit goes out first: the token values of channel / row
    //      i = tid (threads < 128) and the whole checkpoint (16 x 16 B per thread)
    const int i = tid;
    float kt[KC], qt[KC], gt[KC], vt[KC];
    if (tid < kD) {
#pragma unroll
        for (int t = 0; t < KC; ++t) {
            kt[t] = qt[t] = gt[t] = vt[t] = 0.f;
            if (t < ql) {
                const size_t th = ((size_t)r * K + t) * H + h;
                kt[t] = A::load1(k, th * kD + i);
                qt[t] = A::load1(q, th * kD + i);
                gt[t] = A::load1(gate_raw, th * kD + i);
                vt[t] = A::load1(v, th * kD + i);
            }
        }
    }
    const float braw = (tid >= kD && tid - kD < ql)
                           ? A::load1(beta_raw, ((size_t)r * K + (tid - kD)) * H + h) : 0.f;
    const float4* src = reinterpret_cast<const float4*>(pool + ((size_t)slot * H + h) * (kD * kD));
    float4 x[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int u = tid + kVThreads * j;  // 8-float unit: row u >> 4, columns (u & 15) * 8
        x[2 * j] = __ldcs(src + 2 * u);
        x[2 * j + 1] = __ldcs(src + 2 * u + 1);
    }
    if (warp == 0) tmem_alloc(smem_u32(s_tmem), 32);
    if (tid == 0) mbar_init(smem_u32(mbar), 1);
    if (tid >= kD && tid - kD < ql) sbeta[tid - kD] = beta_act(braw, flags);
    if (tid >= kD && tid < kD + 64) {
        // records: key and raw gate exactly as given (upper threads, off the critical path)
        const int e = tid - kD;
        for (int t = 0; t < ql; ++t) {
            const size_t th = ((size_t)r * K + t) * H + h;
            if (e < 32)
                A::copy4(rec_kg, (rec0 + t) * 2 * kD + 4 * e, k, th * kD + 4 * e);
            else
                A::copy4(rec_kg, (rec0 + t) * 2 * kD + kD + 4 * (e - 32), gate_raw, th * kD + 4 * (e - 32));
        }
    }

    // ---- checkpoint S_0^T (rows c, key channels i) -> bf16 hi/lo K-major operand tiles
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int u = tid + kVThreads * j;
        const int c = u >> 4, g = (u & 15) * 8;
        const float e[8] = {x[2 * j].x, x[2 * j].y, x[2 * j].z, x[2 * j].w,
                            x[2 * j + 1].x, x[2 * j + 1].y, x[2 * j + 1].z, x[2 * j + 1].w};
        uint4 hi, lo;
        split8(e, hi, lo);
        *reinterpret_cast<uint4*>(sm + ST_HI + chunk_k(c, g, 128)) = hi;
        *reinterpret_cast<uint4*>(sm + ST_LO + chunk_k(c, g, 128)) = lo;
    }

    // ---- per key channel i: gated keys (rows 0..KC-1) and queries (rows KC..2KC-1) of the
    //      B operand, the records, and the K x K pair factors
    if (tid < kD) {
        float at[KC];
        float cum = 1.f;  // e^{G_t}
        uint16_t* bh = reinterpret_cast<uint16_t*>(sm + KQ_HI);
        uint16_t* bl = reinterpret_cast<uint16_t*>(sm + KQ_LO);
        auto put = [&](int n, float val) {
            const __nv_bfloat16 hh = __float2bfloat16_rn(val);
            const __nv_bfloat16 ll = __float2bfloat16_rn(val - __bfloat162float(hh));
            const uint32_t off = (chunk_k(n, i & ~7, NB) + (i & 7) * 2) >> 1;
            bh[off] = __bfloat16_as_ushort(hh);
            bl[off] = __bfloat16_as_ushort(ll);
        };
#pragma unroll
        for (int t = 0; t < KC; ++t) {
            qt[t] *= scale;
            at[t] = 1.f;
            if (t < ql) {
                at[t] = expf(gate_log(gt[t], flags));
                cum *= at[t];
            }
            put(t, kt[t] * cum);
            put(KC + t, qt[t] * cum);
        }
#pragma unroll
        for (int n = 2 * KC; n < NB; ++n) put(n, 0.f);
        // pair sums over channels, e^{G_t - G_s} as running products of alpha:
        // value [a][b] = P_ab (a <= b) or A_ab (a > b), summed over the warp's 32 channels
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
            int n = NV;
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                const bool upper = (lane & off) != 0;
                const int half = n / 2;
#pragma unroll
                for (int e = 0; e < NV / 2; ++e) {
                    if (e < half) {
                        const float send = upper ? vals[e] : vals[e + half];
                        const float keep = upper ? vals[e + half] : vals[e];
                        vals[e] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                    }
                }
                n = half;
            }
            constexpr int M = NV / 32;
#pragma unroll
            for (int e = 0; e < M; ++e) {
                const int idx = lane * M + e;
                if (idx < KC * KC) red[warp][idx / KC][idx % KC] = vals[e];
            }
        } else {
#pragma unroll
            for (int s0 = 0; s0 < KC; ++s0) {
                if (s0 >= ql) continue;
                float dec = 1.f;
#pragma unroll
                for (int t = s0; t < KC; ++t) {
                    if (t >= ql) continue;
                    if (t > s0) dec *= at[t];
                    const float pp = warp_sum(qt[t] * kt[s0] * dec);
                    if (lane == 0) red[warp][s0][t] = pp;
                    if (t > s0) {
                        const float pa = warp_sum(kt[t] * kt[s0] * dec);
                        if (lane == 0) red[warp][t][s0] = pa;
                    }
                }
            }
        }
    }
    fence_async_smem();
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *s_tmem;
    // ---- D[c][n] = sum_i S_0^T[c][i] B[n][i]: hi*hi + lo*hi + hi*lo
    if (tid == 0) {
        const uint32_t id = idesc_bf16(128, NB, false, false, false);
#pragma unroll
        for (int pass = 0; pass < 3; ++pass) {
            const uint32_t a = sb + (pass == 1 ? ST_LO : ST_HI);
            const uint32_t b = sb + (pass == 2 ? KQ_LO : KQ_HI);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma(tmem, desc_k(a, 128, s), desc_k(b, NB, s), id, (pass | s) != 0);
        }
        commit(smem_u32(mbar));
    }
    for (int e = tid; e < KC * KC; e += kVThreads) {
        const int a = e / KC, b = e - a * KC;
        AP[a][b] = red[0][a][b] + red[1][a][b] + red[2][a][b] + red[3][a][b];
    }
    __syncthreads();
    const bool ok = mbar_wait(smem_u32(mbar), 0, kVWaitLimit);
    fence_after();
    const bool any_timeout = __syncthreads_or(!ok);
    float d[32];
    if (!any_timeout && warp < 4) ld32(tmem + ((uint32_t)(warp * 32) << 16), d);

    // ---- triangular solve for row c, outputs and correction records
    const int c = tid;
    float u[KC];
#pragma unroll
    for (int t = 0; t < KC; ++t) {
        u[t] = 0.f;
        if (t >= K || tid >= kD) continue;
        const size_t th = ((size_t)r * K + t) * H + h;
        if (t < ql && !any_timeout) {
            float acc = d[t];
#pragma unroll
            for (int s0 = 0; s0 < t; ++s0) acc = fmaf(AP[t][s0], u[s0], acc);
            u[t] = sbeta[t] * (vt[t] - acc);
            float o = d[KC + t];
#pragma unroll
            for (int s0 = 0; s0 <= t; ++s0) o = fmaf(AP[s0][t], u[s0], o);
            store1<kBf16Out>(out, th * kD + c, o);
            rec_u[(rec0 + t) * kD + c] = u[t];
        } else {
            store1<kBf16Out>(out, th * kD + c, 0.f);
            rec_u[(rec0 + t) * kD + c] = 0.f;
            if (c < 64) A::zero4(rec_kg, (rec0 + t) * 2 * kD + 4 * c);
        }
    }
    if (any_timeout && tid == 0) report(dev_status, KDA_DEV_TIMEOUT);
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0) tmem_dealloc(tmem, 32);
}

template <int KC>
constexpr size_t verify_smem() {
    constexpr int NB = 2 * KC < 16 ? 16 : 2 * KC;
    return 1024 + 65536 + 2 * NB * 256 + 5 * KC * KC * 4 + KC * 4 + 32;
}

template <int KC, bool I, bool O>
void launch_kc(const void* q, const void* k, const void* v, const void* b, const void* g, int32_t R,
               int32_t K, const int32_t* ql, int32_t H, float scale, uint32_t flags,
               const float* pool, int64_t P, const int32_t* ckpt, float* ru, void* rkg, void* out,
               int32_t* st, cudaStream_t s) {
    constexpr size_t smem = verify_smem<KC>();
    cudaFuncSetAttribute(verify_kernel<KC, I, O>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)smem);
    verify_kernel<KC, I, O><<<(unsigned)(R * H), kVThreads, smem, s>>>(
        q, k, v, b, g, K, ql, H, scale, flags, pool, P, ckpt, ru, rkg, out, st);
}

template <bool I, bool O>
void launch(const void* q, const void* k, const void* v, const void* b, const void* g, int32_t R,
            int32_t K, const int32_t* ql, int32_t H, float scale, uint32_t flags,
            const float* pool, int64_t P, const int32_t* ckpt, float* ru, void* rkg, void* out,
            int32_t* st, cudaStream_t s) {
    if (K <= 2) launch_kc<2, I, O>(q, k, v, b, g, R, K, ql, H, scale, flags, pool, P, ckpt, ru, rkg, out, st, s);
    else if (K <= 4) launch_kc<4, I, O>(q, k, v, b, g, R, K, ql, H, scale, flags, pool, P, ckpt, ru, rkg, out, st, s);
    else if (K <= 8) launch_kc<8, I, O>(q, k, v, b, g, R, K, ql, H, scale, flags, pool, P, ckpt, ru, rkg, out, st, s);
    else launch_kc<16, I, O>(q, k, v, b, g, R, K, ql, H, scale, flags, pool, P, ckpt, ru, rkg, out, st, s);
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" kda_status kda_spec_verify(const void* q, const void* k, const void* v,
                                      const void* beta_raw, const void* gate_raw,
                                      kda_dtype in_dtype, int32_t R, int32_t K,
                                      const int32_t* q_len, int32_t H, int32_t dk, int32_t dv,
                                      float scale, uint32_t flags, const float* state_pool,
                                      int64_t P, const int32_t* ckpt_slot, float* rec_u,
                                      void* rec_kg, void* out, kda_dtype out_dtype,
                                      int32_t* dev_status, void* stream) {
    KDA_REQUIRE(R >= 0 && K >= 0 && H > 0 && P >= 0, KDA_ERR_INVALID_ARG);
    KDA_REQUIRE(dk == kD && dv == kD, KDA_ERR_UNSUPPORTED);
    KDA_REQUIRE(dtype_ok(in_dtype) && dtype_ok(out_dtype), KDA_ERR_UNSUPPORTED);
    KDA_REQUIRE(K <= kMaxVerifyK, KDA_ERR_UNSUPPORTED);
    if (R == 0 || K == 0) return KDA_OK;
    KDA_REQUIRE((int64_t)R * H < (1ll << 31), KDA_ERR_UNSUPPORTED);
    const void* ptrs[] = {q, k, v, beta_raw, gate_raw, state_pool, ckpt_slot, rec_u, rec_kg, out};
    for (const void* p : ptrs) KDA_REQUIRE(p != nullptr && aligned16(p), KDA_ERR_INVALID_ARG);
    cudaStream_t s = as_stream(stream);
    const bool ib = in_dtype == KDA_BF16, ob = out_dtype == KDA_BF16;
    if (ib && ob) launch<true, true>(q, k, v, beta_raw, gate_raw, R, K, q_len, H, scale, flags, state_pool, P, ckpt_slot, rec_u, rec_kg, out, dev_status, s);
    else if (ib) launch<true, false>(q, k, v, beta_raw, gate_raw, R, K, q_len, H, scale, flags, state_pool, P, ckpt_slot, rec_u, rec_kg, out, dev_status, s);
    else if (ob) launch<false, true>(q, k, v, beta_raw, gate_raw, R, K, q_len, H, scale, flags, state_pool, P, ckpt_slot, rec_u, rec_kg, out, dev_status, s);
    else launch<false, false>(q, k, v, beta_raw, gate_raw, R, K, q_len, H, scale, flags, state_pool, P, ckpt_slot, rec_u, rec_kg, out, dev_status, s);
    return launch_status();
}
