// kda_common.cuh -- device helpers shared by the libkda kernels (sm_103a).
//
// Gate and beta activations are applied inside every kernel with the same
// code, in fp32: g = -softplus(raw gate) per key channel, beta = sigmoid(raw
// beta).  The "state semantics" page (section 4) records that prefill and
// decode/verify activated the gate in different places in the engines it
// read; using one device function everywhere removes that difference here.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

constexpr int kD = 128;  // d_k = d_v
constexpr int kChunk = 64;

// ----------------------------------------------------------------------------
// activations (fp32), one form for every kernel
//
// The decay of key channel i at one token is alpha = e^{g}, g = -softplus(x):
// alpha = 1 / (1 + e^x), and 1 / alpha = 1 + e^x.  Every kernel (tensor-core and
// token-serial prefill, decode, verify, commit) takes alpha and 1 / alpha from
// decay_of(), so the same raw gate gives the same alpha bits everywhere: a state
// rebuilt by the commit from a verify record decays exactly as decode decays it.
// e^x is CUDA's __expf and the reciprocal __fdividef(1, .): raw -inf gives
// alpha = 1 exactly; a raw gate above ~88 (e^x = inf) gives alpha = 0.  Under
// KDA_GATE_LOG the input is g itself: alpha = e^g, 1 / alpha = e^{-g}.

struct Decay {
    float a;    // alpha
    float inv;  // 1 / alpha
};

__device__ __forceinline__ Decay decay_of(float raw, uint32_t flags) {
    Decay d;
    if (flags & KDA_GATE_LOG) {
        d.a = __expf(raw);
        d.inv = __expf(-raw);
    } else {
        d.inv = 1.f + __expf(raw);
        d.a = __fdividef(1.f, d.inv);
    }
    return d;
}

__device__ __forceinline__ float alpha_of(float raw, uint32_t flags) { return decay_of(raw, flags).a; }

// Runs body(flags) with the gate form fixed at compile time (KDA_GATE_LOG or not), so that a loop
// of decay_of calls in the body is straight-line code: with the flag tested inside an unrolled
// loop, each element's exponential / reciprocal chain ran after the previous one's branch.  The
// arithmetic is decay_of's either way (the same bits).
template <class Body>
__device__ __forceinline__ void with_gate_form(uint32_t flags, Body&& body) {
    if (flags & KDA_GATE_LOG)
        body(KDA_GATE_LOG);
    else
        body(0u);
}

// Under KDA_QK_L2NORM a row x of q or k is used as x * l2norm_factor(sum_i x_i^2).
constexpr float kL2NormEps = 1e-6f;
__device__ __forceinline__ float l2norm_factor(float sum_sq) { return rsqrtf(sum_sq + kL2NormEps); }

// beta = sigmoid(raw beta) (raw -inf gives 0 exactly); KDA_BETA_ACT: beta given.
__device__ __forceinline__ float beta_act(float raw, uint32_t flags) {
    if (flags & KDA_BETA_ACT) return raw;
    return 1.f / (1.f + expf(-raw));
}

// ----------------------------------------------------------------------------
// element access for bf16 / fp32 activations

template <bool kBf16>
struct Act;

template <>
struct Act<true> {
    using T = __nv_bfloat16;
    // four consecutive elements starting at element index i (i % 4 == 0)
    static __device__ __forceinline__ float4 load4(const void* p, size_t i) {
        const uint2 w = __ldg(reinterpret_cast<const uint2*>(static_cast<const T*>(p) + i));
        float4 r;
        r.x = __uint_as_float(w.x << 16);
        r.y = __uint_as_float(w.x & 0xffff0000u);
        r.z = __uint_as_float(w.y << 16);
        r.w = __uint_as_float(w.y & 0xffff0000u);
        return r;
    }
    static __device__ __forceinline__ float load1(const void* p, size_t i) {
        return __bfloat162float(static_cast<const T*>(p)[i]);
    }
    // raw 8-byte copy of four elements (records keep the input bits)
    static __device__ __forceinline__ void copy4(void* dst, size_t di, const void* src, size_t si) {
        *reinterpret_cast<uint2*>(static_cast<T*>(dst) + di) =
            __ldg(reinterpret_cast<const uint2*>(static_cast<const T*>(src) + si));
    }
    static __device__ __forceinline__ void zero4(void* dst, size_t di) {
        *reinterpret_cast<uint2*>(static_cast<T*>(dst) + di) = make_uint2(0u, 0u);
    }
};

template <>
struct Act<false> {
    static __device__ __forceinline__ float4 load4(const void* p, size_t i) {
        return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p) + i));
    }
    static __device__ __forceinline__ float load1(const void* p, size_t i) {
        return static_cast<const float*>(p)[i];
    }
    static __device__ __forceinline__ void copy4(void* dst, size_t di, const void* src, size_t si) {
        *reinterpret_cast<float4*>(static_cast<float*>(dst) + di) =
            __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(src) + si));
    }
    static __device__ __forceinline__ void zero4(void* dst, size_t di) {
        *reinterpret_cast<float4*>(static_cast<float*>(dst) + di) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// ----------------------------------------------------------------------------
// state element types (pool slots and snapshots): fp32 by default, bf16 or
// fp16 under KDA_STATE_BF16 / KDA_STATE_F16.  Loads widen exactly; a store
// rounds the fp32 value once, to nearest even, straight to the slot's type
// (an fp16 slot never passes through bf16).

enum StateType : int { kStateF32 = 0, kStateBF16 = 1, kStateF16 = 2 };

__host__ __device__ constexpr int state_bytes(int st) { return st == kStateF32 ? 4 : 2; }

__host__ __device__ inline int state_type(uint32_t flags) {
    return (flags & KDA_STATE_BF16) ? kStateBF16 : (flags & KDA_STATE_F16) ? kStateF16 : kStateF32;
}

__host__ __device__ inline bool state_flags_ok(uint32_t flags) {
    return !((flags & KDA_STATE_BF16) && (flags & KDA_STATE_F16));
}

template <int ST>
struct State;

template <>
struct State<kStateF32> {
    // four consecutive elements from element index i (i % 4 == 0); _cs = streaming
    static __device__ __forceinline__ float4 load4(const void* p, size_t i) {
        return *reinterpret_cast<const float4*>(static_cast<const float*>(p) + i);
    }
    static __device__ __forceinline__ float4 load4_cs(const void* p, size_t i) {
        return __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(p) + i));
    }
    static __device__ __forceinline__ void store4(void* p, size_t i, float4 x) {
        *reinterpret_cast<float4*>(static_cast<float*>(p) + i) = x;
    }
    static __device__ __forceinline__ void store4_cs(void* p, size_t i, float4 x) {
        __stcs(reinterpret_cast<float4*>(static_cast<float*>(p) + i), x);
    }
};

template <>
struct State<kStateBF16> {
    static __device__ __forceinline__ float4 widen(uint2 w) {
        return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                           __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
    }
    static __device__ __forceinline__ uint2 narrow(float4 x) {
        __nv_bfloat162 a = __floats2bfloat162_rn(x.x, x.y), b = __floats2bfloat162_rn(x.z, x.w);
        return make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
    }
    static __device__ __forceinline__ float4 load4(const void* p, size_t i) {
        return widen(*reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p) + i));
    }
    static __device__ __forceinline__ float4 load4_cs(const void* p, size_t i) {
        return widen(__ldcs(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p) + i)));
    }
    static __device__ __forceinline__ void store4(void* p, size_t i, float4 x) {
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p) + i) = narrow(x);
    }
    static __device__ __forceinline__ void store4_cs(void* p, size_t i, float4 x) {
        __stcs(reinterpret_cast<uint2*>(static_cast<uint16_t*>(p) + i), narrow(x));
    }
};

template <>
struct State<kStateF16> {
    static __device__ __forceinline__ float4 widen(uint2 w) {
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&w.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&w.y));
        return make_float4(a.x, a.y, b.x, b.y);
    }
    static __device__ __forceinline__ uint2 narrow(float4 x) {
        __half2 a = __floats2half2_rn(x.x, x.y), b = __floats2half2_rn(x.z, x.w);
        return make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
    }
    static __device__ __forceinline__ float4 load4(const void* p, size_t i) {
        return widen(*reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p) + i));
    }
    static __device__ __forceinline__ float4 load4_cs(const void* p, size_t i) {
        return widen(__ldcs(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(p) + i)));
    }
    static __device__ __forceinline__ void store4(void* p, size_t i, float4 x) {
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(p) + i) = narrow(x);
    }
    static __device__ __forceinline__ void store4_cs(void* p, size_t i, float4 x) {
        __stcs(reinterpret_cast<uint2*>(static_cast<uint16_t*>(p) + i), narrow(x));
    }
};

// runtime-typed forms for the sites off the hot loops (initial / final states, snapshots)
__device__ __forceinline__ float4 state_load4(const void* p, size_t i, int st) {
    if (st == kStateBF16) return State<kStateBF16>::load4(p, i);
    if (st == kStateF16) return State<kStateF16>::load4(p, i);
    return State<kStateF32>::load4(p, i);
}

__device__ __forceinline__ void state_store4(void* p, size_t i, float4 x, int st) {
    if (st == kStateBF16) State<kStateBF16>::store4(p, i, x);
    else if (st == kStateF16) State<kStateF16>::store4(p, i, x);
    else State<kStateF32>::store4(p, i, x);
}

// element offset of (slot, head) in a pool of 128 x 128 states, as a byte pointer
__host__ __device__ inline size_t state_elem(int64_t slot, int H, int h) {
    return ((size_t)slot * H + h) * (size_t)(kD * kD);
}

template <bool kBf16Out>
__device__ __forceinline__ void store1(void* out, size_t i, float x) {
    if constexpr (kBf16Out)
        static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(x);
    else
        static_cast<float*>(out)[i] = x;
}

template <bool kBf16Out>
__device__ __forceinline__ void store4(void* out, size_t i, float4 x) {
    if constexpr (kBf16Out) {
        uint2 w = make_uint2(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w));
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + i) = w;
    } else {
        *reinterpret_cast<float4*>(static_cast<float*>(out) + i) = x;
    }
}

__device__ __forceinline__ void report(int32_t* dev_status, int32_t bits) {
    if (dev_status) atomicOr(dev_status, bits);
}

// Accepted length of one speculative request from the verify step's input ids
// and the target's sampled ids (the request's rows start at `row`): 1 + the
// number of leading drafts tokens[i+1] equal to sampled[i], so 1 <= a <= q_len;
// 0 when q_len = 0 and -1 when q_len lies outside [0, K].  Warp-collective:
// all 32 lanes call it for the same request; K <= 32, and no id at or past
// q_len is read.
__device__ __forceinline__ int accepted_length(const int32_t* __restrict__ tokens,
                                               const int32_t* __restrict__ sampled, size_t row,
                                               int ql, int K, int lane) {
    if (ql < 0 || ql > K) return -1;
    if (ql == 0) return 0;
    // lane < ql - 1 implies lane + 1 < ql <= K; lane ql - 1 <= 31 always counts as a miss
    const bool miss = lane >= ql - 1 || tokens[row + lane + 1] != sampled[row + lane];
    return __ffs(__ballot_sync(0xffffffffu, miss));
}

// Short-convolution tensors of one call (descriptors by value in the kernel parameters).
struct ConvDescs {
    kda_conv_desc d[KDA_MAX_POOLS];
};

// One thread's 16-byte column of a conv slot: rows a .. a+keep-1 move to rows 0 .. keep-1
// (a >= 1), in groups of up to 8 with every read of a group before its writes; later groups
// read rows a+j.. >= j+1, above every row written so far, so overlapping ranges are safe.
__device__ __forceinline__ void conv_move_rows(uint8_t* col, int64_t row_bytes, int a, int keep) {
    for (int j = 0; j < keep; j += 8) {
        const int n = keep - j < 8 ? keep - j : 8;
        uint4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (q < n) v[q] = __ldcs(reinterpret_cast<const uint4*>(col + (int64_t)(a + j + q) * row_bytes));
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (q < n) __stcs(reinterpret_cast<uint4*>(col + (int64_t)(j + q) * row_bytes), v[q]);
    }
}

// Checks of one (tensor, request) of a conv compaction; true when rows must move.  Reports
// a bad slot / accepted length once per pair (lead thread).
__device__ __forceinline__ bool conv_pair_ok(const kda_conv_desc& c, int s, int a, int keep,
                                             bool lead, int32_t* dev_status) {
    if (s < 0) return false;
    if (s >= c.num_slots) {
        if (lead) report(dev_status, KDA_DEV_BAD_SLOT);
        return false;
    }
    if (a < 0 || a + keep > c.n_rows) {
        if (lead) report(dev_status, KDA_DEV_BAD_ACCEPT);
        return false;
    }
    return a > 0;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Sum two values across the warp with interleaved shuffles.
__device__ __forceinline__ void warp_sum2(float& a, float& b) {
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        b += __shfl_xor_sync(0xffffffffu, b, o);
    }
}

// Elementwise products and FMAs in packed fp32 pairs (each lane rounds as the scalar
// operation does, so results are the scalar ones; half the instructions issue).
__device__ __forceinline__ float4 f4_mul(float4 a, float4 b) {
    const float2 lo = __fmul2_rn(make_float2(a.x, a.y), make_float2(b.x, b.y));
    const float2 hi = __fmul2_rn(make_float2(a.z, a.w), make_float2(b.z, b.w));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}
__device__ __forceinline__ float f4_dot(float4 a, float4 b) {
    return fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, a.w * b.w)));
}
__device__ __forceinline__ float4 f4_fma(float s, float4 k, float4 x) {
    const float2 ss = make_float2(s, s);
    const float2 lo = __ffma2_rn(ss, make_float2(k.x, k.y), make_float2(x.x, x.y));
    const float2 hi = __ffma2_rn(ss, make_float2(k.z, k.w), make_float2(x.z, x.w));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
}

// ----------------------------------------------------------------------------
// One recurrence step for 16 state rows held by a warp.
//
// The warp holds S^T rows [row0, row0+16) (a row = one value channel, 128 key
// channels); lane l owns key channels [4l, 4l+4).  For each row c:
//   x = alpha (.) S^T[c]              (X = Diag(alpha) S, by key channel)
//   u = beta (v[c] - x . k)
//   S^T[c] = x + u k
//   o[c] = scale (x . q + u (k . q))  (= S_t^T (scale q))
// Returns u and o of row c in lane (c - row0) (other lanes get garbage).
struct StepIn {
    float4 a;   // alpha for this lane's 4 key channels
    float4 k;
    float4 q;   // already multiplied by scale
    float kq;   // full k . q (scaled)
    float beta;
};

template <int RW>
__device__ __forceinline__ void step_rows(float4 (&s)[RW], const StepIn& in, const float (&vrow)[RW],
                                          float& u_mine, float& o_mine, int lane) {
#pragma unroll
    for (int r = 0; r < RW; ++r) {
        float4 x = f4_mul(s[r], in.a);
        float d1 = f4_dot(x, in.k);
        float d2 = f4_dot(x, in.q);
        warp_sum2(d1, d2);
        const float u = in.beta * (vrow[r] - d1);
        s[r] = f4_fma(u, in.k, x);
        const float o = fmaf(u, in.kq, d2);
        if (lane == r) {
            u_mine = u;
            o_mine = o;
        }
    }
}

// ----------------------------------------------------------------------------
// A tile of consecutive token rows staged in shared memory with the
// activations applied: alpha = exp(g), q scaled, beta activated, k . q.
template <int kTile>
struct TokenTile {
    float a[kTile][kD];
    float k[kTile][kD];
    float q[kTile][kD];
    float v[kTile][kD];
    float beta[kTile];
    float kq[kTile];
};

// Rows row_base .. row_base+n_tok-1 of head h; 8 warps, a warp per row.
template <bool kBf16, int kTile>
__device__ __forceinline__ void stage_tokens(TokenTile<kTile>& tt, const void* q, const void* k,
                                             const void* v, const void* beta_raw,
                                             const void* gate_raw, size_t row_base, int n_tok,
                                             int H, int h, float scale, uint32_t flags) {
    using A = Act<kBf16>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int t = warp; t < n_tok; t += (int)(blockDim.x >> 5)) {
        const size_t th = (row_base + t) * (size_t)H + h;
        const float4 g = A::load4(gate_raw, th * kD + 4 * lane);
        float4 kk = A::load4(k, th * kD + 4 * lane);
        const float4 qq = A::load4(q, th * kD + 4 * lane);
        const float4 vv = A::load4(v, th * kD + 4 * lane);
        const float4 a = make_float4(alpha_of(g.x, flags), alpha_of(g.y, flags),
                                     alpha_of(g.z, flags), alpha_of(g.w, flags));
        float fk = 1.f, fq = scale;
        if (flags & KDA_QK_L2NORM) {
            float sk = f4_dot(kk, kk), sq = f4_dot(qq, qq);
            warp_sum2(sk, sq);
            fk = l2norm_factor(sk);
            fq = scale * l2norm_factor(sq);
        }
        kk = make_float4(kk.x * fk, kk.y * fk, kk.z * fk, kk.w * fk);
        const float4 qs = make_float4(qq.x * fq, qq.y * fq, qq.z * fq, qq.w * fq);
        *reinterpret_cast<float4*>(&tt.a[t][4 * lane]) = a;
        *reinterpret_cast<float4*>(&tt.k[t][4 * lane]) = kk;
        *reinterpret_cast<float4*>(&tt.q[t][4 * lane]) = qs;
        *reinterpret_cast<float4*>(&tt.v[t][4 * lane]) = vv;
        const float kq = warp_sum(f4_dot(kk, qs));
        if (lane == 0) {
            tt.kq[t] = kq;
            tt.beta[t] = beta_act(A::load1(beta_raw, th), flags);
        }
    }
}

// Recurrence step for token t of a staged tile on the warp's 16 rows.
template <int kTile>
__device__ __forceinline__ void step_from_tile(float4 (&s)[16], const TokenTile<kTile>& tt, int t,
                                               int row0, int lane, float& u_m, float& o_m) {
    StepIn in;
    in.a = *reinterpret_cast<const float4*>(&tt.a[t][4 * lane]);
    in.k = *reinterpret_cast<const float4*>(&tt.k[t][4 * lane]);
    in.q = *reinterpret_cast<const float4*>(&tt.q[t][4 * lane]);
    in.kq = tt.kq[t];
    in.beta = tt.beta[t];
    float vrow[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 x = *reinterpret_cast<const float4*>(&tt.v[t][row0 + 4 * i]);
        vrow[4 * i] = x.x;
        vrow[4 * i + 1] = x.y;
        vrow[4 * i + 2] = x.z;
        vrow[4 * i + 3] = x.w;
    }
    step_rows<16>(s, in, vrow, u_m, o_m, lane);
}

}  // namespace kda
