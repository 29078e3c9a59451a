// prefill_api.cu -- host entry point of kda_chunk_prefill: argument checks and
// kernel selection.
#include "kda_common.cuh"
#include "kda_host.h"
#include "prefill.h"

using namespace kda;

extern "C" size_t kda_chunk_prefill_workspace_size(int32_t T_tot, int32_t N, int32_t H,
                                                   int32_t dk, int32_t dv, int32_t chunk) {
    (void)dk;
    (void)dv;
    (void)chunk;
    const size_t two_phase = prefill_2p_workspace(T_tot, N, H);
    const size_t single = prefill_tc_workspace(N);
    return two_phase > single ? two_phase : single;
}

extern "C" kda_status kda_chunk_prefill(const void* q, const void* k, const void* v,
                                        const void* beta_raw, const void* gate_raw,
                                        kda_dtype in_dtype, const int32_t* cu_seqlens, int32_t N,
                                        int32_t T_tot, int32_t H, int32_t dk, int32_t dv,
                                        int32_t chunk, float scale, uint32_t flags,
                                        void* state_pool, int64_t P, const int32_t* init_slot,
                                        const int32_t* final_slot, const int32_t* track_chunk_idx,
                                        int32_t M, void* track_state, void* out,
                                        kda_dtype out_dtype, void* workspace, size_t ws_bytes,
                                        int32_t* dev_status, void* stream) {
    KDA_REQUIRE(N >= 0 && T_tot >= 0 && H > 0 && P >= 0 && M >= 0, KDA_ERR_INVALID_ARG);
    KDA_REQUIRE(dk == kD && dv == kD && chunk == kChunk, KDA_ERR_UNSUPPORTED);
    KDA_REQUIRE(dtype_ok(in_dtype) && dtype_ok(out_dtype), KDA_ERR_UNSUPPORTED);
    KDA_REQUIRE(M <= kMaxTrack, KDA_ERR_UNSUPPORTED);
    KDA_REQUIRE(state_flags_ok(flags), KDA_ERR_UNSUPPORTED);
    KDA_REQUIRE((int64_t)N * H < (1ll << 31), KDA_ERR_UNSUPPORTED);
    if (N == 0) return KDA_OK;
    KDA_REQUIRE(cu_seqlens != nullptr && aligned16(cu_seqlens), KDA_ERR_INVALID_ARG);
    if (T_tot > 0) {
        const void* ptrs[] = {q, k, v, beta_raw, gate_raw, out};
        for (const void* p : ptrs) KDA_REQUIRE(p != nullptr && aligned16(p), KDA_ERR_INVALID_ARG);
    }
    if (init_slot || final_slot) KDA_REQUIRE(state_pool != nullptr && aligned16(state_pool), KDA_ERR_INVALID_ARG);
    if (M > 0) {
        KDA_REQUIRE(track_chunk_idx != nullptr && track_state != nullptr, KDA_ERR_INVALID_ARG);
        KDA_REQUIRE(aligned16(track_chunk_idx) && aligned16(track_state), KDA_ERR_INVALID_ARG);
    }
    if (workspace) KDA_REQUIRE(aligned16(workspace), KDA_ERR_INVALID_ARG);
    PrefillArgs p{q,     k,         v,         beta_raw,   gate_raw,        cu_seqlens, N,
                  T_tot, H,         scale,     flags,      state_pool,      P,          init_slot,
                  final_slot, track_chunk_idx, M, track_state, out, dev_status, state_type(flags)};
    const bool bf16_in = in_dtype == KDA_BF16, bf16_out = out_dtype == KDA_BF16;
    const bool chunked = !(flags & KDA_PREFILL_RECURRENT);
    const size_t ws_2p = prefill_2p_workspace(T_tot, N, H);
    if (chunked && prefill_2p_supported(p) && workspace && ws_2p > 0 && ws_bytes >= ws_2p)
        return launch_prefill_2p(p, bf16_in, bf16_out, workspace, as_stream(stream));
    if (chunked && prefill_tc_supported(p, bf16_in))
        launch_prefill_tc(p, bf16_out, workspace, ws_bytes, as_stream(stream));
    else
        launch_prefill_serial(p, bf16_in, bf16_out, as_stream(stream));
    return launch_status();
}
