// prefill.h -- arguments shared by the kda_chunk_prefill kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

constexpr int kMaxTrack = 1024;  // snapshot requests per sequence
constexpr int kMaxOrderN = 4096; // sequences ordered longest-first by the tensor-core prefill

struct PrefillArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* beta_raw;
    const void* gate_raw;
    const int32_t* cu_seqlens;
    int32_t N, T_tot, H;
    float scale;
    uint32_t flags;
    void* pool;  // states of type st (pool slots and snapshots alike)
    int64_t P;
    const int32_t* init_slot;
    const int32_t* final_slot;
    const int32_t* track;
    int32_t M;
    void* track_state;
    void* out;
    int32_t* dev_status;
    int32_t st;  // StateType of pool and track_state
};

void launch_prefill_serial(const PrefillArgs& p, bool bf16_in, bool bf16_out, cudaStream_t s);

// the two-phase kernels take bf16 or fp32 activations and either output type
bool prefill_2p_supported(const PrefillArgs& p);
size_t prefill_2p_workspace(int32_t T_tot, int32_t N, int32_t H);
kda_status launch_prefill_2p(const PrefillArgs& p, bool bf16_in, bool bf16_out, void* workspace, cudaStream_t s);

bool prefill_tc_supported(const PrefillArgs& p, bool bf16_in);
size_t prefill_tc_workspace(int32_t N);
void launch_prefill_tc(const PrefillArgs& p, bool bf16_out, void* workspace, size_t ws_bytes,
                       cudaStream_t s);

}  // namespace kda
