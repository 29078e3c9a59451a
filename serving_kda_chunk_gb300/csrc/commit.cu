// commit.cu -- kda_spec_commit: commit plan + closed-form state rebuild at
// the accepted length.
//
// vLLM PR 51855 page (RecoverSSM), implementation breakdown item 4: after
// sampling, a plan step derives the accepted lengths on the GPU and the commit
// rebuilds the state at the accepted position in reverse order in one shot
// instead of re-running the recursion.  With the records of verify (u_t fp32,
// k_t and the raw gate in the activation dtype), for accepted length a:
//     S_a = Diag(exp c_0) S_0 + sum_{t=1..a} Diag(exp c_t) k_t u_t^T,
//     c_t = sum_{t<s<=a} g_s  (c_0 = sum_{s<=a} g_s),
// so every state element is one fused sum of a+1 terms.
//
// Each CTA owns 16 KiB of one (request, head) state: 32 rows of S^T in fp32
// (four CTAs per state) or 64 rows of 16-bit states (two).  Every load of a
// CTA is issued up front with cp.async into shared memory, so the bytes in
// flight cost no registers: its checkpoint rows, the a key / raw-gate records
// (one contiguous block) and its rows of u_t.  Threads then walk the records
// backwards per key channel to form F_t = exp(c_t) k_t and the total decay
// exp(c_0) as running products of alpha = exp(g) = 1 / (1 + e^x), and each
// warp updates its rows four at a time and streams them to the destination
// slot (in place allowed: the checkpoint rows were staged before any store).
#include <type_traits>

#include "kda_common.cuh"
#include "kda_host.h"
#include "umma.cuh"

namespace kda {
namespace {

constexpr int kMaxCommitK = 32;  // a request's records fit in shared memory beside the staged rows

constexpr int kCommitThreads = 128;  // 4 warps
constexpr int kCommitStage = 16384;  // bytes of checkpoint rows per CTA, staged by cp.async
// state rows per warp: 8 fp32 rows (a quarter of a state per CTA) or 16 rows of 16-bit
// states (half a state per CTA)
template <int ST>
__host__ __device__ constexpr int commit_rows() { return kCommitStage / (4 * kD * state_bytes(ST)); }
template <int ST>
__host__ __device__ constexpr int commit_ctas() { return kD / (4 * commit_rows<ST>()); }

// Accepted lengths: read from num_accepted, or (kTokens) found by every warp
// of every CTA from the request's token ids, with the lengths and next tokens
// written out once per request.
struct AcceptArgs {
    const int32_t* acc;      // [R] accepted lengths (plain commit)
    const int32_t* tokens;   // [R, K] verify input ids (kTokens)
    const int32_t* sampled;  // [R, K] sampled ids (kTokens)
    int32_t* acc_out;        // [R] or null (kTokens)
    int32_t* next_out;       // [R] or null (kTokens)
};

// Short-convolution windows moved in the same launch (kTokens only): n_ctas blocks at the
// front of the grid, gy per (tensor, request), each a 128-chunk column range of the rows.
struct ConvArgs {
    ConvDescs convs;
    int32_t n_convs;
    const int32_t* slot;  // [R] conv slot of each request
    int32_t keep;
    int32_t gy;
    int32_t n_ctas;       // 0: no conv work
};

// Align mode (kTokens only): the state at the last block boundary inside each accepted span.
struct AlignArgs {
    const int32_t* seq_len0;   // [R] tokens before the step; null: no align work
    const int32_t* block_slot; // [R] slot receiving the boundary state, or null
    int32_t* block_idx_out;    // [R] floor((seq_len0 + a) / block_size), or null
    int32_t block_size;
};

template <bool kBf16Rec, bool kTokens, int ST>
__global__ void __launch_bounds__(kCommitThreads, 8) commit_kernel(
    void* __restrict__ pool, int64_t P, const int32_t* __restrict__ ckpt,
    const int32_t* __restrict__ dst, const AcceptArgs acc_args, const ConvArgs conv,
    const AlignArgs align,
    const int32_t* __restrict__ q_len, int32_t K, int32_t H, uint32_t flags,
    const float* __restrict__ rec_u, const void* __restrict__ rec_kg, int32_t* __restrict__ plan_out,
    int32_t* __restrict__ dev_status) {
    constexpr int ES = kBf16Rec ? 2 : 4;  // record element size
    constexpr int RW = commit_rows<ST>(), CR = 4 * RW, CU = commit_ctas<ST>();  // rows / warp, CTA
    extern __shared__ __align__(16) float sm[];
    uint8_t* STG = reinterpret_cast<uint8_t*>(sm);          // [CR][128] checkpoint rows
    float* F = sm + kCommitStage / 4;                       // [K][128]
    float* U = F + K * kD;                                  // [K][CR] this CTA's rows of u_t
    float* D = U + K * CR;                                  // [128]
    uint8_t* KG = reinterpret_cast<uint8_t*>(D + kD);       // [K][256] raw records (k, gate)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if constexpr (kTokens) {
        if ((int)blockIdx.x < conv.n_ctas) {  // a conv block: its request's window only
            const int pair = blockIdx.x / conv.gy, y = blockIdx.x - pair * conv.gy;
            const int i = pair % conv.n_convs, rc = pair / conv.n_convs;
            const kda_conv_desc c = conv.convs.d[i];
            const int qlc = q_len ? q_len[rc] : K;
            const int ac = accepted_length(acc_args.tokens, acc_args.sampled, (size_t)rc * K, qlc, K, lane);
            const int sc = conv.slot[rc];
            if (!conv_pair_ok(c, sc, ac, conv.keep, threadIdx.x == 0 && y == 0, dev_status)) return;
            const int64_t chunk = (int64_t)y * kCommitThreads + threadIdx.x;
            if (chunk < c.row_bytes / 16)
                conv_move_rows(static_cast<uint8_t*>(c.base) + (int64_t)sc * c.slot_stride_bytes + chunk * 16,
                               c.row_bytes, ac, conv.keep);
            return;
        }
    }
    const int bid = blockIdx.x - (kTokens ? conv.n_ctas : 0);
    const int unit = bid / CU;  // (request, head); the rest picks the row block
    const int part = bid - unit * CU;
    const int r = unit / H, h = unit - r * H;
    const int row0 = part * CR + warp * RW;
    const int src = ckpt[r];
    const int d = dst ? dst[r] : src;
    const int ql = q_len ? q_len[r] : K;
    int a;
    if constexpr (kTokens)
        a = accepted_length(acc_args.tokens, acc_args.sampled, (size_t)r * K, ql, K, lane);
    else
        a = acc_args.acc[r];
    const bool slot_ok = src >= 0 && src < P && d >= 0 && d < P;
    const bool ok = slot_ok && ql >= 0 && ql <= K && a >= 0 && a <= ql;
    int a_b = -1, bslot = -1;  // align mode: accepted length ending on a block boundary, its slot
    if constexpr (kTokens) {
        if (align.seq_len0) {
            const int L0 = align.seq_len0[r];
            const bool valid = L0 >= 0 && a >= 0;
            const int hi = valid ? (int)(((int64_t)L0 + a) / align.block_size) : -1;
            if (valid && hi > L0 / align.block_size) {
                a_b = (int)((int64_t)hi * align.block_size - L0);
                bslot = align.block_slot ? align.block_slot[r] : -1;
            }
            if (h == 0 && part == 0 && threadIdx.x == 0) {
                if (align.block_idx_out) align.block_idx_out[r] = hi;
                if (ok && bslot >= P) report(dev_status, KDA_DEV_BAD_SLOT);
            }
            if (bslot >= P) bslot = -1;
        }
    }
    if (h == 0 && part == 0 && threadIdx.x == 0) {
        if constexpr (kTokens) {
            if (acc_args.acc_out) acc_args.acc_out[r] = a;
            if (acc_args.next_out)
                acc_args.next_out[r] = a > 0 ? acc_args.sampled[(size_t)r * K + a - 1] : -1;
        }
        if (plan_out) {
            plan_out[3 * r + 0] = ok ? a : -1;
            plan_out[3 * r + 1] = src;
            plan_out[3 * r + 2] = d;
        }
        if (!ok) report(dev_status, slot_ok ? KDA_DEV_BAD_ACCEPT : KDA_DEV_BAD_SLOT);
    }
    if (!ok) return;
    using SIO = State<ST>;
    const size_t S0 = state_elem(src, H, h), SD = state_elem(d, H, h);
    if (a == 0) {
        if (d == src) return;
#pragma unroll 4
        for (int i = 0; i < RW; ++i) {
            // a 16-bit value widens and rounds back to itself: the copy is exact
            const float4 x = SIO::load4_cs(pool, S0 + (size_t)(row0 + i) * kD + 4 * lane);
            SIO::store4_cs(pool, SD + (size_t)(row0 + i) * kD + 4 * lane, x);
        }
        return;
    }
    // every load up front, into shared memory: checkpoint rows, key / raw-gate records, u rows
    const size_t rec0 = ((size_t)r * H + h) * K;
    {
        const uint32_t stg_s = umma::smem_u32(STG), kg_s = umma::smem_u32(KG), u_s = umma::smem_u32(U);
        const uint8_t* s0_g = static_cast<const uint8_t*>(pool) + (S0 + (size_t)part * CR * kD) * state_bytes(ST);
#pragma unroll
        for (int e = threadIdx.x; e < kCommitStage / 16; e += kCommitThreads)
            umma::cp_async16(stg_s + 16 * e, s0_g + 16 * e, 16);
        const uint8_t* kg_g = static_cast<const uint8_t*>(rec_kg) + rec0 * 2 * kD * ES;
        for (int e = threadIdx.x; e < a * 2 * kD * ES / 16; e += kCommitThreads)
            umma::cp_async16(kg_s + 16 * e, kg_g + 16 * e, 16);
        // u_t rows part*CR .. part*CR+CR-1: CR/4 chunks of 16 B per step
        constexpr int kChunks = CR / 4;
        for (int e = threadIdx.x; e < a * kChunks; e += kCommitThreads) {
            const int t = e / kChunks, ch = e - t * kChunks;
            umma::cp_async16(u_s + (uint32_t)(t * CR * 4 + ch * 16),
                             rec_u + (rec0 + t) * kD + part * CR + ch * 4, 16);
        }
        umma::cp_async_commit();
    }
    umma::cp_async_wait_all();
    // KDA_QK_L2NORM: the record holds k as given; its factor per step (a warp per record)
    float* NRM = reinterpret_cast<float*>(KG + (size_t)K * 2 * kD * ES);  // [K]
    const bool l2 = (flags & KDA_QK_L2NORM) != 0;
    if (l2) {
        __syncthreads();  // every thread's record copies have landed
        for (int t = warp; t < a; t += kCommitThreads / 32) {
            float4 x;
            if constexpr (kBf16Rec)
                x = State<kStateBF16>::widen(*reinterpret_cast<const uint2*>(KG + ((size_t)t * 2 * kD + 4 * lane) * 2));
            else
                x = *reinterpret_cast<const float4*>(KG + ((size_t)t * 2 * kD + 4 * lane) * 4);
            const float ss = warp_sum(f4_dot(x, x));
            if (lane == 0) NRM[t] = l2norm_factor(ss);
        }
    }
    // pass 0: the state after a steps -> the destination slot; pass 1 (align mode): the state
    // after a_b steps -> the block slot.  The staged checkpoint rows are only read.
    const int n_pass = bslot >= 0 ? 2 : 1;
#pragma unroll 1
    for (int pass = 0; pass < n_pass; ++pass) {
        const int aa = pass ? a_b : a;
        const size_t dst_elem = pass ? state_elem(bslot, H, h) : SD;
        __syncthreads();  // staging landed / the previous pass finished with F and D
        {
            // F_t = k_t exp(c_t), c_t = sum over s in (t, aa) of g_s: a running product of alpha
            // from t = aa - 1 down; D = exp(c_0 + g_0) = the product over the aa steps
            const int c = threadIdx.x;
            float prod = 1.f;
            with_gate_form(flags, [&](uint32_t form) {
                for (int t = aa - 1; t >= 0; --t) {
                    const float kv = kBf16Rec ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(KG)[t * 2 * kD + c] << 16)
                                              : reinterpret_cast<const float*>(KG)[t * 2 * kD + c];
                    const float gv = kBf16Rec ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(KG)[t * 2 * kD + kD + c] << 16)
                                              : reinterpret_cast<const float*>(KG)[t * 2 * kD + kD + c];
                    F[t * kD + c] = prod * (l2 ? kv * NRM[t] : kv);
                    prod *= alpha_of(gv, form);
                }
            });
            D[c] = prod;
        }
        __syncthreads();
        const float4 dec = *reinterpret_cast<const float4*>(&D[4 * lane]);
        // this warp's rows in groups of 4 (row = index within the CTA's staged block)
#pragma unroll
        for (int g4 = 0; g4 < RW; g4 += 4) {
            const int rb = warp * RW + g4;
            float4 s[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float4 x;
                if constexpr (ST == kStateF32)
                    x = *reinterpret_cast<const float4*>(STG + (rb + i) * 512 + lane * 16);
                else
                    x = SIO::widen(*reinterpret_cast<const uint2*>(STG + (rb + i) * 256 + lane * 8));
                s[i] = f4_mul(x, dec);
            }
            for (int t = 0; t < aa; ++t) {
                const float4 f = *reinterpret_cast<const float4*>(&F[t * kD + 4 * lane]);
                const float4 u0 = *reinterpret_cast<const float4*>(&U[t * CR + rb]);
                s[0] = f4_fma(u0.x, f, s[0]);
                s[1] = f4_fma(u0.y, f, s[1]);
                s[2] = f4_fma(u0.z, f, s[2]);
                s[3] = f4_fma(u0.w, f, s[3]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
                SIO::store4_cs(pool, dst_elem + (size_t)(part * CR + rb + i) * kD + 4 * lane, s[i]);
        }
    }
}

// Host checks and the launch shared by both commit entry points.
kda_status launch_commit(void* state_pool, int64_t P, const int32_t* ckpt_slot,
                         const int32_t* dst_slot, const AcceptArgs& acc, const ConvArgs& conv,
                         const AlignArgs& align, bool from_tokens,
                         const int32_t* q_len, int32_t R, int32_t K, int32_t H, int32_t dk,
                         int32_t dv, uint32_t flags, const float* rec_u, const void* rec_kg,
                         kda_dtype rec_dtype, int32_t* plan_out, int32_t* dev_status,
                         void* stream) {
    KDA_REQUIRE(R >= 0 && K >= 0 && H > 0 && P >= 0, KDA_ERR_INVALID_ARG);
    KDA_REQUIRE(dk == kD && dv == kD, KDA_ERR_UNSUPPORTED);
    KDA_REQUIRE(dtype_ok(rec_dtype), KDA_ERR_UNSUPPORTED);
    KDA_REQUIRE(K <= kMaxCommitK, KDA_ERR_UNSUPPORTED);
    KDA_REQUIRE(state_flags_ok(flags), KDA_ERR_UNSUPPORTED);
    if (R == 0) return KDA_OK;
    KDA_REQUIRE((int64_t)R * H < (1ll << 30), KDA_ERR_UNSUPPORTED);
    const void* ptrs[] = {state_pool, ckpt_slot, rec_u, rec_kg};
    for (const void* p : ptrs) KDA_REQUIRE(p != nullptr && aligned16(p), KDA_ERR_INVALID_ARG);
    if (from_tokens) {
        KDA_REQUIRE(K >= 1, KDA_ERR_INVALID_ARG);
        const void* tok[] = {acc.tokens, acc.sampled};
        for (const void* p : tok) KDA_REQUIRE(p != nullptr && aligned16(p), KDA_ERR_INVALID_ARG);
        const void* opt[] = {acc.acc_out, acc.next_out};
        for (const void* p : opt) KDA_REQUIRE(p == nullptr || aligned16(p), KDA_ERR_INVALID_ARG);
    } else {
        KDA_REQUIRE(acc.acc != nullptr && aligned16(acc.acc), KDA_ERR_INVALID_ARG);
    }
    cudaStream_t s = as_stream(stream);
    const size_t es = rec_dtype == KDA_BF16 ? 2 : 4;
    const int st = state_type(flags);
    const int rows = st == kStateF32 ? 4 * commit_rows<kStateF32>() : 4 * commit_rows<kStateBF16>();
    const size_t smem = kCommitStage + (size_t)(K * kD + K * rows + kD) * sizeof(float) +
                        (size_t)K * 2 * kD * es + (size_t)((K + 3) / 4) * 16;  // + L2 factors
    const unsigned grid = (unsigned)((kD / rows) * R * H + conv.n_ctas);
    auto run = [&](auto kernel) {
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        kernel<<<grid, kCommitThreads, smem, s>>>(state_pool, P, ckpt_slot, dst_slot, acc, conv,
                                                  align, q_len, K, H, flags, rec_u, rec_kg,
                                                  plan_out, dev_status);
    };
    auto by_state = [&](auto rec_bf16, auto tokens) {
        constexpr bool B = decltype(rec_bf16)::value, T = decltype(tokens)::value;
        switch (st) {
            case kStateBF16: run(commit_kernel<B, T, kStateBF16>); break;
            case kStateF16: run(commit_kernel<B, T, kStateF16>); break;
            default: run(commit_kernel<B, T, kStateF32>);
        }
    };
    using yes = std::true_type;
    using no = std::false_type;
    if (rec_dtype == KDA_BF16)
        from_tokens ? by_state(yes{}, yes{}) : by_state(yes{}, no{});
    else
        from_tokens ? by_state(no{}, yes{}) : by_state(no{}, no{});
    return launch_status();
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" kda_status kda_spec_commit(void* state_pool, int64_t P, const int32_t* ckpt_slot,
                                      const int32_t* dst_slot, const int32_t* num_accepted,
                                      const int32_t* q_len, int32_t R, int32_t K, int32_t H,
                                      int32_t dk, int32_t dv, uint32_t flags, const float* rec_u,
                                      const void* rec_kg, kda_dtype rec_dtype, int32_t* plan_out,
                                      int32_t* dev_status, void* stream) {
    const AcceptArgs acc{num_accepted, nullptr, nullptr, nullptr, nullptr};
    const ConvArgs conv{};
    const AlignArgs align{};
    return launch_commit(state_pool, P, ckpt_slot, dst_slot, acc, conv, align, false, q_len, R, K,
                         H, dk, dv, flags, rec_u, rec_kg, rec_dtype, plan_out, dev_status, stream);
}

extern "C" kda_status kda_spec_accept_commit(
    void* state_pool, int64_t P, const int32_t* ckpt_slot, const int32_t* dst_slot,
    const int32_t* tokens, const int32_t* sampled, const int32_t* q_len, int32_t R, int32_t K,
    int32_t H, int32_t dk, int32_t dv, uint32_t flags, const float* rec_u, const void* rec_kg,
    kda_dtype rec_dtype, int32_t* num_accepted, int32_t* next_token, int32_t* plan_out,
    const kda_commit_extras* extras, int32_t* dev_status, void* stream) {
    const AcceptArgs acc{nullptr, tokens, sampled, num_accepted, next_token};
    ConvArgs conv{};
    AlignArgs align{};
    const kda_commit_extras none{};
    const kda_commit_extras& x = extras ? *extras : none;
    KDA_REQUIRE(x.n_convs >= 0 && x.n_convs <= KDA_MAX_POOLS, KDA_ERR_INVALID_ARG);
    if (x.n_convs > 0 && R > 0) {
        KDA_REQUIRE(x.convs != nullptr && x.conv_keep >= 1, KDA_ERR_INVALID_ARG);
        KDA_REQUIRE(x.conv_slot != nullptr && aligned16(x.conv_slot), KDA_ERR_INVALID_ARG);
        int64_t max_chunks = 0;
        for (int i = 0; i < x.n_convs; ++i) {
            const kda_conv_desc& c = x.convs[i];
            KDA_REQUIRE(c.base != nullptr && aligned16(c.base), KDA_ERR_INVALID_ARG);
            KDA_REQUIRE(c.row_bytes > 0 && c.row_bytes % 16 == 0, KDA_ERR_INVALID_ARG);
            KDA_REQUIRE(c.n_rows >= x.conv_keep && c.num_slots > 0, KDA_ERR_INVALID_ARG);
            KDA_REQUIRE(c.slot_stride_bytes % 16 == 0 && c.slot_stride_bytes >= c.n_rows * c.row_bytes,
                        KDA_ERR_INVALID_ARG);
            conv.convs.d[i] = c;
            if (c.row_bytes / 16 > max_chunks) max_chunks = c.row_bytes / 16;
        }
        const int64_t gy = (max_chunks + kCommitThreads - 1) / kCommitThreads;
        KDA_REQUIRE((int64_t)R * x.n_convs * gy < (1ll << 30), KDA_ERR_UNSUPPORTED);
        conv.n_convs = x.n_convs;
        conv.slot = x.conv_slot;
        conv.keep = x.conv_keep;
        conv.gy = (int32_t)gy;
        conv.n_ctas = (int32_t)(R * x.n_convs * gy);
    }
    if (x.seq_len0 != nullptr) {
        // a span of at most K accepted positions crosses at most one boundary only when
        // block_size >= K; smaller blocks are the configuration the align path cannot serve
        KDA_REQUIRE(x.block_size > 0, KDA_ERR_INVALID_ARG);
        KDA_REQUIRE(x.block_size >= K, KDA_ERR_UNSUPPORTED);
        const void* opt[] = {x.seq_len0, x.block_slot, x.block_idx_out};
        for (const void* p : opt) KDA_REQUIRE(p == nullptr || aligned16(p), KDA_ERR_INVALID_ARG);
        align = AlignArgs{x.seq_len0, x.block_slot, x.block_idx_out, x.block_size};
    }
    return launch_commit(state_pool, P, ckpt_slot, dst_slot, acc, conv, align, true, q_len, R, K,
                         H, dk, dv, flags, rec_u, rec_kg, rec_dtype, plan_out, dev_status, stream);
}
