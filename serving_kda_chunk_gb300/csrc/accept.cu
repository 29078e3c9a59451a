// accept.cu -- kda_spec_accept: the accepted length of every speculative
// request, computed on the device from token ids.
//
// vLLM PR 51855 page (RecoverSSM), implementation breakdown item 4: after
// sampling, the commit plan derives each request's runtime accepted length on
// the GPU and writes num_accepted_tokens back to device buffers, so that the
// commit that follows needs no host round trip.  Position 0 of a request holds
// its last committed token and positions 1..q_len-1 its drafts; sampled[i] is
// the target model's token for the position after i.  Draft i+1 is kept while
// it equals sampled[i], and the state keeps the updates of the committed token
// plus every kept draft: a = 1 + kept, and the next input is sampled[a-1].
//
// One warp per request: lane i compares draft i+1 with sampled token i, a
// ballot marks the mismatches (lanes at or past the last draft count as one),
// and the lowest set bit gives a directly.  K <= 32 keeps a request in one warp.
// kda_spec_accept_commit runs the same warp step at the head of every commit CTA.
#include "kda_common.cuh"
#include "kda_host.h"

namespace kda {
namespace {

constexpr int kMaxAcceptK = 32;
constexpr int kAcceptWarps = 4;

__global__ void __launch_bounds__(kAcceptWarps * 32) accept_kernel(
    const int32_t* __restrict__ tokens, const int32_t* __restrict__ sampled,
    const int32_t* __restrict__ q_len, int32_t R, int32_t K, int32_t* __restrict__ num_accepted,
    int32_t* __restrict__ next_token, int32_t* __restrict__ dev_status) {
    const int r = blockIdx.x * kAcceptWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (r >= R) return;  // uniform across the warp
    const int ql = q_len ? q_len[r] : K;
    const size_t row = (size_t)r * K;
    const int a = accepted_length(tokens, sampled, row, ql, K, lane);
    if (lane == 0) {
        if (a < 0) report(dev_status, KDA_DEV_BAD_ACCEPT);
        num_accepted[r] = a;
        if (next_token) next_token[r] = a > 0 ? sampled[row + a - 1] : -1;
    }
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" kda_status kda_spec_accept(const int32_t* tokens, const int32_t* sampled,
                                      const int32_t* q_len, int32_t R, int32_t K,
                                      int32_t* num_accepted, int32_t* next_token,
                                      int32_t* dev_status, void* stream) {
    KDA_REQUIRE(R >= 0 && K >= 1, KDA_ERR_INVALID_ARG);
    KDA_REQUIRE(K <= kMaxAcceptK, KDA_ERR_UNSUPPORTED);
    if (R == 0) return KDA_OK;
    const void* ptrs[] = {tokens, sampled, num_accepted};
    for (const void* p : ptrs) KDA_REQUIRE(p != nullptr && aligned16(p), KDA_ERR_INVALID_ARG);
    const void* opt[] = {q_len, next_token};
    for (const void* p : opt) KDA_REQUIRE(p == nullptr || aligned16(p), KDA_ERR_INVALID_ARG);
    const unsigned grid = (unsigned)((R + kAcceptWarps - 1) / kAcceptWarps);
    accept_kernel<<<grid, kAcceptWarps * 32, 0, as_stream(stream)>>>(
        tokens, sampled, q_len, R, K, num_accepted, next_token, dev_status);
    return launch_status();
}
