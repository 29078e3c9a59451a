// decode.cu -- kda_recurrent_decode: one token per request, in place over a
// slot-indexed state pool (fp32, or bf16 / fp16 slots widened on load and
// rounded once on store).
//
// "State semantics" page, section 4: decode applies the gate activation inside
// the kernel and updates the per-head state in place.
//
// A CTA of 4 warps owns 16 KiB of one (request, head) state: 32 rows of S^T in
// fp32 or 64 rows of 16-bit states (a row = one value channel, 128 contiguous
// key channels).  The whole block is requested at once with cp.async into
// shared memory, so the bytes in flight cost no registers and many CTAs per SM
// keep HBM busy; the token's activations load meanwhile.  Each warp then walks
// its rows (a lane owns 4 key channels) and writes each updated row straight
// back to the slot with streaming stores.  With fp32 rows the two row dot
// products of a row are one interleaved warp reduction; 16-bit rows, half the
// bytes for the same arithmetic, are issue-bound, so there the eight dot
// products of four rows are reduce-scattered across the warp in 14 shuffles
// instead of 40 (the same pairwise sums, so the same bits).  Bound by HBM traffic: 2 x the state per
// (request, head).
#include "kda_common.cuh"
#include "kda_host.h"
#include "umma.cuh"

namespace kda {
namespace {

constexpr int kDecThreads = 128;       // 4 warps
constexpr int kDecStage = 16384;       // bytes of state per CTA

template <int ST>
__host__ __device__ constexpr int dec_rows() { return kDecStage / (kD * state_bytes(ST)); }  // per CTA
template <int ST>
__host__ __device__ constexpr int dec_ctas() { return kD / dec_rows<ST>(); }  // per (request, head)

template <int ST>
__device__ __forceinline__ float4 smem_row4(const uint8_t* buf, int row, int lane) {
    if constexpr (ST == kStateF32) {
        return *reinterpret_cast<const float4*>(buf + row * 512 + lane * 16);
    } else {
        const uint2 w = *reinterpret_cast<const uint2*>(buf + row * 256 + lane * 8);
        return State<ST>::widen(w);
    }
}

template <bool kBf16In, bool kBf16Out, int ST>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(
    const void* __restrict__ q, const void* __restrict__ k, const void* __restrict__ v,
    const void* __restrict__ beta_raw, const void* __restrict__ gate_raw, int32_t H, float scale,
    uint32_t flags, void* __restrict__ pool, int64_t P, const int32_t* __restrict__ slots,
    void* __restrict__ out, int32_t* __restrict__ dev_status) {
    using A = Act<kBf16In>;
    using SIO = State<ST>;
    constexpr int CR = dec_rows<ST>(), CU = dec_ctas<ST>(), RW = CR / 4;  // rows per CTA / warp
    __shared__ __align__(16) uint8_t buf[kDecStage];
    const int unit = blockIdx.x / CU;
    const int part = blockIdx.x - unit * CU;
    const int r = unit / H, h = unit - r * H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t th = (size_t)r * H + h;
    const int slot = slots[r];
    if (slot < 0 || slot >= P) {
        if (slot >= P && threadIdx.x == 0 && part == 0) report(dev_status, KDA_DEV_BAD_SLOT);
        if (threadIdx.x < CR / 4)
            store4<kBf16Out>(out, th * kD + part * CR + 4 * threadIdx.x, make_float4(0.f, 0.f, 0.f, 0.f));
        return;
    }
    const size_t S = state_elem(slot, H, h) + (size_t)part * CR * kD;  // this CTA's first row
    {
        const uint8_t* src = static_cast<const uint8_t*>(pool) + S * state_bytes(ST);
        const uint32_t dst = umma::smem_u32(buf);
#pragma unroll
        for (int e = threadIdx.x; e < kDecStage / 16; e += kDecThreads)
            umma::cp_async16(dst + 16 * e, src + 16 * e, 16);
        umma::cp_async_commit();
    }
    StepIn in;
    const float4 g = A::load4(gate_raw, th * kD + 4 * lane);
    in.a = make_float4(alpha_of(g.x, flags), alpha_of(g.y, flags), alpha_of(g.z, flags),
                       alpha_of(g.w, flags));
    in.k = A::load4(k, th * kD + 4 * lane);
    float4 qq = A::load4(q, th * kD + 4 * lane);
    float fq = scale;
    if (flags & KDA_QK_L2NORM) {  // per (row, head), over the 128 channels the warp holds
        float sk = f4_dot(in.k, in.k), sq = f4_dot(qq, qq);
        warp_sum2(sk, sq);
        const float fk = l2norm_factor(sk);
        fq = scale * l2norm_factor(sq);
        in.k = make_float4(in.k.x * fk, in.k.y * fk, in.k.z * fk, in.k.w * fk);
    }
    in.q = make_float4(qq.x * fq, qq.y * fq, qq.z * fq, qq.w * fq);
    in.kq = warp_sum(f4_dot(in.k, in.q));
    in.beta = beta_act(A::load1(beta_raw, th), flags);
    const int row0 = warp * RW;  // within the CTA's rows
    if constexpr (ST == kStateF32) {
        // one row at a time: the two row dot products are one interleaved warp reduction
        const float vm = lane < RW ? A::load1(v, th * kD + part * CR + row0 + lane) : 0.f;
        umma::cp_async_wait_all();
        __syncthreads();
        float o_m = 0.f;
#pragma unroll 4
        for (int i = 0; i < RW; ++i) {
            const float4 x = f4_mul(smem_row4<ST>(buf, row0 + i, lane), in.a);
            float d1 = f4_dot(x, in.k), d2 = f4_dot(x, in.q);
            warp_sum2(d1, d2);
            const float u = in.beta * (__shfl_sync(0xffffffffu, vm, i) - d1);
            SIO::store4_cs(pool, S + (size_t)(row0 + i) * kD + 4 * lane, f4_fma(u, in.k, x));
            if (lane == i) o_m = fmaf(u, in.kq, d2);
        }
        if (lane < RW) store1<kBf16Out>(out, th * kD + part * CR + row0 + lane, o_m);
    } else {
        // 16-bit rows carry half the bytes for the same arithmetic, so the issue rate binds:
        // rows in groups of four.  The eight partial row dot products of a group (d1 = x . k and
        // d2 = x . q of each row) are reduce-scattered across the warp: after halving steps over
        // lane bits 4, 3 and 2 and full sums over bits 1 and 0, lane l holds the total of value
        // m = l >> 2, i.e. d1 of row m (m < 4) or d2 of row m - 4.  u is formed where its d1 is and
        // broadcast for the row update; o is formed where its d2 is.
        const int m = lane >> 2;
        float vloc[RW / 4];  // v of row 4 g + m at the lanes that form u (m < 4)
#pragma unroll
        for (int g = 0; g < RW / 4; ++g)
            vloc[g] = m < 4 ? A::load1(v, th * kD + part * CR + row0 + 4 * g + m) : 0.f;
        umma::cp_async_wait_all();
        __syncthreads();
#pragma unroll
        for (int g = 0; g < RW / 4; ++g) {
            const int rg = row0 + 4 * g;
            float4 x[4];
            float vals[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                x[i] = f4_mul(smem_row4<ST>(buf, rg + i, lane), in.a);
                vals[i] = f4_dot(x[i], in.k);
                vals[4 + i] = f4_dot(x[i], in.q);
            }
#pragma unroll
            for (int step = 0; step < 3; ++step) {  // offsets 16, 8, 4: 8 -> 4 -> 2 -> 1 values
                const int off = 16 >> step, half = 4 >> step;
                const bool upper = (lane & off) != 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (e < half) {
                        const float send = upper ? vals[e] : vals[e + half];
                        const float keep = upper ? vals[e + half] : vals[e];
                        vals[e] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                    }
                }
            }
            float tot = vals[0];
            tot += __shfl_xor_sync(0xffffffffu, tot, 2);
            tot += __shfl_xor_sync(0xffffffffu, tot, 1);
            const float u_here = in.beta * (vloc[g] - tot);  // u of row m at lanes with m < 4
            float uu[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) uu[i] = __shfl_sync(0xffffffffu, u_here, 4 * i);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                SIO::store4_cs(pool, S + (size_t)(rg + i) * kD + 4 * lane, f4_fma(uu[i], in.k, x[i]));
            const float u_o = __shfl_sync(0xffffffffu, u_here, 4 * (m & 3));  // u of row m - 4
            if (m >= 4 && (lane & 3) == 0)
                store1<kBf16Out>(out, th * kD + part * CR + rg + (m - 4), fmaf(u_o, in.kq, tot));
        }
    }
}

template <bool I, bool O>
void launch(const void* q, const void* k, const void* v, const void* b, const void* g, int32_t R,
            int32_t H, float scale, uint32_t flags, void* pool, int64_t P, const int32_t* slot,
            void* out, int32_t* st, cudaStream_t s) {
    const unsigned units = (unsigned)(R * H);
    switch (state_type(flags)) {
        case kStateBF16:
            decode_kernel<I, O, kStateBF16><<<dec_ctas<kStateBF16>() * units, kDecThreads, 0, s>>>(
                q, k, v, b, g, H, scale, flags, pool, P, slot, out, st);
            break;
        case kStateF16:
            decode_kernel<I, O, kStateF16><<<dec_ctas<kStateF16>() * units, kDecThreads, 0, s>>>(
                q, k, v, b, g, H, scale, flags, pool, P, slot, out, st);
            break;
        default:
            decode_kernel<I, O, kStateF32><<<dec_ctas<kStateF32>() * units, kDecThreads, 0, s>>>(
                q, k, v, b, g, H, scale, flags, pool, P, slot, out, st);
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
    KDA_REQUIRE((int64_t)R * H * dec_ctas<kStateF32>() < (1ll << 31), KDA_ERR_UNSUPPORTED);
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
