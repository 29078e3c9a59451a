// decode.cu -- kda_recurrent_decode: one token per request, in place over a
// slot-indexed state pool (fp32, or bf16 / fp16 slots widened on load and
// rounded once on store).
//
// "State semantics" page, section 4: decode applies the gate activation inside
// the kernel and updates the per-head state in place.
//
// Four CTAs per (request, head); their 4 warps each own 8 rows of S^T (a row =
// one value channel, 128 contiguous key channels), a lane owns 4 key channels.
// A CTA's 16 KiB of state is loaded with 16-byte loads before any arithmetic,
// the row dot products are warp reductions, and the updated rows are written
// back in place; small CTAs keep many independent load chains resident.  The kernel is bound by HBM
// traffic: 2 x 64 KiB of fp32 state per (request, head), half that for 16-bit states.
#include "kda_common.cuh"
#include "kda_host.h"

namespace kda {
namespace {

constexpr int kDecThreads = 128;                   // 4 warps
constexpr int kDecRows = 8;                        // state rows per warp
constexpr int kDecCtas = kD / (4 * kDecRows);      // CTAs per (request, head)

template <bool kBf16In, bool kBf16Out, int ST>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(
    const void* __restrict__ q, const void* __restrict__ k, const void* __restrict__ v,
    const void* __restrict__ beta_raw, const void* __restrict__ gate_raw, int32_t H, float scale,
    uint32_t flags, void* __restrict__ pool, int64_t P, const int32_t* __restrict__ slots,
    void* __restrict__ out, int32_t* __restrict__ dev_status) {
    using A = Act<kBf16In>;
    using SIO = State<ST>;
    const int unit = blockIdx.x / kDecCtas;
    const int part = blockIdx.x - unit * kDecCtas;
    const int r = unit / H, h = unit - r * H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = part * (4 * kDecRows) + warp * kDecRows;
    const size_t th = (size_t)r * H + h;
    const int slot = slots[r];
    if (slot < 0 || slot >= P) {
        if (slot >= P && threadIdx.x == 0 && part == 0) report(dev_status, KDA_DEV_BAD_SLOT);
        if (threadIdx.x < 4 * kDecRows / 4)
            store4<kBf16Out>(out, th * kD + part * 4 * kDecRows + 4 * threadIdx.x,
                             make_float4(0.f, 0.f, 0.f, 0.f));
        return;
    }
    const size_t S = state_elem(slot, H, h);
    float4 s[kDecRows];
#pragma unroll
    for (int i = 0; i < kDecRows; ++i) s[i] = SIO::load4_cs(pool, S + (size_t)(row0 + i) * kD + 4 * lane);

    StepIn in;
    const float4 g = A::load4(gate_raw, th * kD + 4 * lane);
    in.a = make_float4(expf(gate_log(g.x, flags)), expf(gate_log(g.y, flags)),
                       expf(gate_log(g.z, flags)), expf(gate_log(g.w, flags)));
    in.k = A::load4(k, th * kD + 4 * lane);
    float4 qq = A::load4(q, th * kD + 4 * lane);
    in.q = make_float4(qq.x * scale, qq.y * scale, qq.z * scale, qq.w * scale);
    in.kq = warp_sum(f4_dot(in.k, in.q));
    in.beta = beta_act(A::load1(beta_raw, th), flags);
    float vrow[kDecRows];
    {
        const float vm = lane < kDecRows ? A::load1(v, th * kD + row0 + lane) : 0.f;
#pragma unroll
        for (int i = 0; i < kDecRows; ++i) vrow[i] = __shfl_sync(0xffffffffu, vm, i);
    }
    float u_m = 0.f, o_m = 0.f;
    step_rows<kDecRows>(s, in, vrow, u_m, o_m, lane);
#pragma unroll
    for (int i = 0; i < kDecRows; ++i) SIO::store4_cs(pool, S + (size_t)(row0 + i) * kD + 4 * lane, s[i]);
    if (lane < kDecRows) store1<kBf16Out>(out, th * kD + row0 + lane, o_m);
}

template <bool I, bool O>
void launch(const void* q, const void* k, const void* v, const void* b, const void* g, int32_t R,
            int32_t H, float scale, uint32_t flags, void* pool, int64_t P, const int32_t* slot,
            void* out, int32_t* st, cudaStream_t s) {
    const unsigned grid = (unsigned)(kDecCtas * R * H);
    switch (state_type(flags)) {
        case kStateBF16:
            decode_kernel<I, O, kStateBF16><<<grid, kDecThreads, 0, s>>>(q, k, v, b, g, H, scale, flags, pool, P, slot, out, st);
            break;
        case kStateF16:
            decode_kernel<I, O, kStateF16><<<grid, kDecThreads, 0, s>>>(q, k, v, b, g, H, scale, flags, pool, P, slot, out, st);
            break;
        default:
            decode_kernel<I, O, kStateF32><<<grid, kDecThreads, 0, s>>>(q, k, v, b, g, H, scale, flags, pool, P, slot, out, st);
    }
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" kda_status kda_recurrent_decode(const void* q, const void* k, const void* v,
                                           const void* beta_raw, const void* gate_raw,
                                           kda_dtype in_dtype, int32_t R, int32_t H, int32_t dk,
                                           int32_t dv, float scale, uint32_t flags,
                                           void* state_pool, int64_t P, const int32_t* slot,
                                           void* out, kda_dtype out_dtype, int32_t* dev_status,
                                           void* stream) {
    KDA_REQUIRE(R >= 0 && H > 0 && P >= 0, KDA_ERR_INVALID_ARG);
    KDA_REQUIRE(dk == kD && dv == kD, KDA_ERR_UNSUPPORTED);
    KDA_REQUIRE(dtype_ok(in_dtype) && dtype_ok(out_dtype), KDA_ERR_UNSUPPORTED);
    KDA_REQUIRE(state_flags_ok(flags), KDA_ERR_UNSUPPORTED);
    if (R == 0) return KDA_OK;
    KDA_REQUIRE((int64_t)R * H * kDecCtas < (1ll << 31), KDA_ERR_UNSUPPORTED);
    const void* ptrs[] = {q, k, v, beta_raw, gate_raw, state_pool, slot, out};
    for (const void* p : ptrs) KDA_REQUIRE(p != nullptr && aligned16(p), KDA_ERR_INVALID_ARG);
    cudaStream_t s = as_stream(stream);
    const bool ib = in_dtype == KDA_BF16, ob = out_dtype == KDA_BF16;
    if (ib && ob) launch<true, true>(q, k, v, beta_raw, gate_raw, R, H, scale, flags, state_pool, P, slot, out, dev_status, s);
    else if (ib) launch<true, false>(q, k, v, beta_raw, gate_raw, R, H, scale, flags, state_pool, P, slot, out, dev_status, s);
    else if (ob) launch<false, true>(q, k, v, beta_raw, gate_raw, R, H, scale, flags, state_pool, P, slot, out, dev_status, s);
    else launch<false, false>(q, k, v, beta_raw, gate_raw, R, H, scale, flags, state_pool, P, slot, out, dev_status, s);
    return launch_status();
}
