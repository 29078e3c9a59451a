// prefill_serial.cu -- token-serial evaluation of kda_chunk_prefill on CUDA
// cores.  It is the simple, precision-first form of the prefill: the same
// recurrence as decode applied token after token with the fp32 state held in
// registers, and the fp32 snapshot written at each requested chunk boundary.
// The tensor-core chunked kernel (prefill_tc.cu) is checked against it on the
// GPU, and it serves shapes the chunked kernel does not take.
//
// SGLang PR 34820 page, implementation breakdown item 2 and the Helion kernel
// listing: while walking a sequence chunk by chunk, the fp32 state accumulator
// itself is written into the snapshot buffer when the chunk index equals the
// sequence's track_chunk_idx; the reading used here is that index j names the
// state after exactly j*chunk tokens of the sequence (the state entering chunk
// j), the convention of per-chunk state stores.
#include "kda_common.cuh"
#include "kda_host.h"
#include "prefill.h"

namespace kda {
namespace {

constexpr int kTok = 16;

template <bool kBf16In, bool kBf16Out>
__global__ void __launch_bounds__(256) prefill_serial_kernel(PrefillArgs p) {
    __shared__ TokenTile<kTok> tt;
    __shared__ int trk[kMaxTrack];
    const int n = blockIdx.x / p.H, h = blockIdx.x - (blockIdx.x / p.H) * p.H;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row0 = warp * 16;
    const int t0 = p.cu_seqlens[n], t1 = p.cu_seqlens[n + 1];
    if (t0 < 0 || t1 < t0 || t1 > p.T_tot || (n == 0 && t0 != 0)) {
        if (threadIdx.x == 0 && h == 0) report(p.dev_status, KDA_DEV_BAD_SEQLEN);
        return;
    }
    const int L = t1 - t0;
    const int n_chunks = (L + kChunk - 1) / kChunk;
    const int init = p.init_slot ? p.init_slot[n] : -1;
    const int fin = p.final_slot ? p.final_slot[n] : -1;
    if (init >= p.P || fin >= p.P) {
        if (threadIdx.x == 0 && h == 0) report(p.dev_status, KDA_DEV_BAD_SLOT);
        return;
    }
    for (int m = threadIdx.x; m < p.M; m += blockDim.x) {
        const int j = p.track[(size_t)n * p.M + m];
        if (j < -1 || j >= n_chunks) {
            if (h == 0) report(p.dev_status, KDA_DEV_BAD_TRACK);
            trk[m] = -1;
        } else {
            trk[m] = j;
        }
    }
    float4 s[16];
    if (init >= 0) {
        const size_t S = state_elem(init, p.H, h);
#pragma unroll
        for (int i = 0; i < 16; ++i) s[i] = state_load4(p.pool, S + (size_t)(row0 + i) * kD + 4 * lane, p.st);
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) s[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    for (int base = 0; base < L; base += kTok) {
        const int nt = min(kTok, L - base);
        __syncthreads();
        stage_tokens<kBf16In, kTok>(tt, p.q, p.k, p.v, p.beta_raw, p.gate_raw, (size_t)t0 + base, nt,
                                    p.H, h, p.scale, p.flags);
        __syncthreads();
        for (int i = 0; i < nt; ++i) {
            const int local = base + i;
            if ((local & (kChunk - 1)) == 0) {
                const int j = local / kChunk;
                for (int m = 0; m < p.M; ++m) {
                    if (trk[m] != j) continue;
                    const size_t snap = state_elem((int64_t)n * p.M + m, p.H, h);
#pragma unroll
                    for (int r = 0; r < 16; ++r)
                        state_store4(p.track_state, snap + (size_t)(row0 + r) * kD + 4 * lane, s[r], p.st);
                }
            }
            float u_m = 0.f, o_m = 0.f;
            step_from_tile(s, tt, i, row0, lane, u_m, o_m);
            if (lane < 16)
                store1<kBf16Out>(p.out, ((size_t)(t0 + local) * p.H + h) * kD + row0 + lane, o_m);
        }
    }
    if (fin >= 0) {
        const size_t S = state_elem(fin, p.H, h);
#pragma unroll
        for (int i = 0; i < 16; ++i) state_store4(p.pool, S + (size_t)(row0 + i) * kD + 4 * lane, s[i], p.st);
    }
}

}  // namespace

void launch_prefill_serial(const PrefillArgs& p, bool bf16_in, bool bf16_out, cudaStream_t s) {
    const unsigned grid = (unsigned)(p.N * p.H);
    if (bf16_in && bf16_out) prefill_serial_kernel<true, true><<<grid, 256, 0, s>>>(p);
    else if (bf16_in) prefill_serial_kernel<true, false><<<grid, 256, 0, s>>>(p);
    else if (bf16_out) prefill_serial_kernel<false, true><<<grid, 256, 0, s>>>(p);
    else prefill_serial_kernel<false, false><<<grid, 256, 0, s>>>(p);
}

}  // namespace kda
