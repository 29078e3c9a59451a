// conv_compact.cu -- kda_conv_compact: the short-convolution window kept after
// a speculative step, on every conv state tensor of the layer in one launch.
//
// vLLM PR 51855 page (RecoverSSM), implementation breakdown item 4: after the
// accepted lengths are known, the commit compacts the convolution history;
// the serving pages describe the conv state as a sliding window moved by an
// offset copy, unlike the recurrent state's whole-block copy.  A slot holds
// `keep` history rows followed by the step's input rows; after a accepted
// positions rows a .. a+keep-1 become rows 0 .. keep-1, the last `keep`
// inputs of the accepted stream.  A draftless request (q_len = 1) takes the
// same path with a = 1.
//
// Grid: one CTA column per (tensor, request), CTAs along y cover the row in
// 16-byte chunks, a thread owns one chunk of every row.  Rows move front to
// back in groups of up to eight, all reads of a group before its writes (the
// reads overlap in flight): every later read is of a row above every row
// written so far, so overlapping ranges (a < keep) are safe without staging.
#include "kda_common.cuh"
#include "kda_host.h"

namespace kda {
namespace {

constexpr int kConvThreads = 256;

__global__ void __launch_bounds__(kConvThreads) conv_compact_kernel(
    const ConvDescs convs, int32_t n_convs, const int32_t* __restrict__ slots,
    const int32_t* __restrict__ acc, int32_t keep, int32_t* __restrict__ dev_status) {
    const int i = blockIdx.x % n_convs, r = blockIdx.x / n_convs;
    const kda_conv_desc c = convs.d[i];
    const int s = slots[r], a = acc[r];
    if (!conv_pair_ok(c, s, a, keep, threadIdx.x == 0 && blockIdx.y == 0, dev_status)) return;
    const int64_t chunk = (int64_t)blockIdx.y * kConvThreads + threadIdx.x;
    if (chunk >= c.row_bytes / 16) return;
    conv_move_rows(static_cast<uint8_t*>(c.base) + (int64_t)s * c.slot_stride_bytes + chunk * 16,
                   c.row_bytes, a, keep);
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" kda_status kda_conv_compact(const kda_conv_desc* convs, int32_t n_convs,
                                       const int32_t* slot, const int32_t* num_accepted,
                                       int32_t R, int32_t keep, int32_t* dev_status,
                                       void* stream) {
    KDA_REQUIRE(convs != nullptr && n_convs > 0 && n_convs <= KDA_MAX_POOLS, KDA_ERR_INVALID_ARG);
    KDA_REQUIRE(R >= 0 && keep >= 1, KDA_ERR_INVALID_ARG);
    ConvDescs d{};
    int64_t max_chunks = 0;
    for (int i = 0; i < n_convs; ++i) {
        const kda_conv_desc& c = convs[i];
        KDA_REQUIRE(c.base != nullptr && aligned16(c.base), KDA_ERR_INVALID_ARG);
        KDA_REQUIRE(c.row_bytes > 0 && c.row_bytes % 16 == 0, KDA_ERR_INVALID_ARG);
        KDA_REQUIRE(c.n_rows >= keep && c.num_slots > 0, KDA_ERR_INVALID_ARG);
        KDA_REQUIRE(c.slot_stride_bytes % 16 == 0 && c.slot_stride_bytes >= c.n_rows * c.row_bytes,
                    KDA_ERR_INVALID_ARG);
        d.d[i] = c;
        if (c.row_bytes / 16 > max_chunks) max_chunks = c.row_bytes / 16;
    }
    if (R == 0) return KDA_OK;
    const void* ptrs[] = {slot, num_accepted};
    for (const void* p : ptrs) KDA_REQUIRE(p != nullptr && aligned16(p), KDA_ERR_INVALID_ARG);
    const int64_t gy = (max_chunks + kConvThreads - 1) / kConvThreads;
    KDA_REQUIRE((int64_t)R * n_convs < (1ll << 31) && gy < 65536, KDA_ERR_UNSUPPORTED);
    conv_compact_kernel<<<dim3((unsigned)(R * n_convs), (unsigned)gy), kConvThreads, 0,
                          as_stream(stream)>>>(d, n_convs, slot, num_accepted, keep, dev_status);
    return launch_status();
}
