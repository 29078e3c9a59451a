// verify.cu -- kda_spec_verify: speculative verify from one checkpoint per
// request, recording what the commit needs.
//
// vLLM PR 51855 page (RecoverSSM), implementation breakdown items 1 and 3:
// verify only reads the checkpoint, computes the output at each speculative
// position and writes the fp32 correction u and the activation-dtype key and
// raw gate into per-request record buffers of shape (heads, positions, d) and
// (heads, positions, 2 d).
//
// One CTA per (request, head).  The checkpoint is read once into registers
// (8 warps x 16 rows of S^T, 4 key channels per lane) and never written; the
// K positions' inputs are staged in shared memory with the activations
// applied, then stepped through in order.
#include "kda_common.cuh"
#include "kda_host.h"

namespace kda {
namespace {

constexpr int kVerifyTile = 8;

template <bool kBf16In, bool kBf16Out>
__global__ void __launch_bounds__(256) verify_kernel(
    const void* __restrict__ q, const void* __restrict__ k, const void* __restrict__ v,
    const void* __restrict__ beta_raw, const void* __restrict__ gate_raw, int32_t K,
    const int32_t* __restrict__ q_len, int32_t H, float scale, uint32_t flags,
    const float* __restrict__ pool, int64_t P, const int32_t* __restrict__ ckpt,
    float* __restrict__ rec_u, void* __restrict__ rec_kg, void* __restrict__ out,
    int32_t* __restrict__ dev_status) {
    using A = Act<kBf16In>;
    __shared__ TokenTile<kVerifyTile> tt;
    const int unit = blockIdx.x;
    const int r = unit / H, h = unit - r * H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = warp * 16;
    const int slot = ckpt[r];
    int ql = q_len ? q_len[r] : K;
    const bool slot_ok = slot >= 0 && slot < P;
    const bool len_ok = ql >= 0 && ql <= K;
    if (!(slot_ok && len_ok)) {
        if (threadIdx.x == 0 && h == 0) {
            if (slot >= P) report(dev_status, KDA_DEV_BAD_SLOT);
            if (!len_ok) report(dev_status, KDA_DEV_BAD_ACCEPT);
        }
        ql = 0;
    }
    float4 s[16];
    if (ql > 0) {
        const float* S = pool + ((size_t)slot * H + h) * (kD * kD);
#pragma unroll
        for (int i = 0; i < 16; ++i)
            s[i] = __ldcs(reinterpret_cast<const float4*>(S + (size_t)(row0 + i) * kD) + lane);
    }
    for (int t0 = 0; t0 < K; t0 += kVerifyTile) {
        const int n_live = min(kVerifyTile, ql - t0);
        if (n_live > 0) {
            __syncthreads();
            stage_tokens<kBf16In, kVerifyTile>(tt, q, k, v, beta_raw, gate_raw, (size_t)r * K + t0,
                                               n_live, H, h, scale, flags);
            __syncthreads();
        }
        const int n_here = min(kVerifyTile, K - t0);
        for (int i = 0; i < n_here; ++i) {
            const int t = t0 + i;
            const size_t th = ((size_t)r * K + t) * H + h;
            const size_t rec = ((size_t)r * H + h) * K + t;
            if (t < ql) {
                float u_m = 0.f, o_m = 0.f;
                step_from_tile(s, tt, i, row0, lane, u_m, o_m);
                if (lane < 16) {
                    store1<kBf16Out>(out, th * kD + row0 + lane, o_m);
                    rec_u[rec * kD + row0 + lane] = u_m;
                }
                if (warp == 0) A::copy4(rec_kg, rec * 2 * kD + 4 * lane, k, th * kD + 4 * lane);
                if (warp == 1)
                    A::copy4(rec_kg, rec * 2 * kD + kD + 4 * lane, gate_raw, th * kD + 4 * lane);
            } else {
                if (lane < 16) {
                    store1<kBf16Out>(out, th * kD + row0 + lane, 0.f);
                    rec_u[rec * kD + row0 + lane] = 0.f;
                }
                if (warp < 2) A::zero4(rec_kg, rec * 2 * kD + warp * kD + 4 * lane);
            }
        }
    }
}

template <bool I, bool O>
void launch(const void* q, const void* k, const void* v, const void* b, const void* g, int32_t R,
            int32_t K, const int32_t* ql, int32_t H, float scale, uint32_t flags,
            const float* pool, int64_t P, const int32_t* ckpt, float* ru, void* rkg, void* out,
            int32_t* st, cudaStream_t s) {
    verify_kernel<I, O><<<(unsigned)(R * H), 256, 0, s>>>(q, k, v, b, g, K, ql, H, scale, flags,
                                                          pool, P, ckpt, ru, rkg, out, st);
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
