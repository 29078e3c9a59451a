// prefill_2p.cu -- two-phase chunked KDA prefill: a parallel prep over every
// (chunk, head), then one sequential sweep per (sequence, head).
//
// The chunk form of the recurrence (G_t = sum_{u<=t} g_u inside the chunk, per key channel):
//   A_ts = sum_i k_ti k_si e^{G_ti - G_si} (s < t),  P_ts = sum_i q_ti k_si e^{G_ti - G_si} (s <= t)
//   T    = (I + Diag(beta) A)^-1,   T_b = T Diag(beta),   W = T_b (k e^{G})
//   U    = T_b V - W S,             O   = (q e^{G}) S + P U
//   S   <- Diag(e^{G_63}) S + (k e^{G_63 - G})^T U
// Everything left of "S" depends on the chunk's own inputs only.  The prep kernel computes it
// for all (chunk, head) pairs at once -- gates, A and P (tcgen05), the triangular solve, T_b,
// W (tcgen05), the decayed query / key operands -- and writes each pair's operands to a
// workspace block, already laid out as the sweep's shared-memory MMA tiles.  The sweep kernel
// then walks one (sequence, head) chunk by chunk with the fp32 state resident in TMEM and runs
// only the state-dependent products; it fetches each block with two bulk (TMA) copies.
//
// Why two phases.  The state recurrence puts a sequence's chunks in series, and the
// state-independent half of a chunk is most of its latency (the gate products, the 64 x 64
// solve, the operand splits).  A single pass keeps that half on the serial path of each
// (sequence, head) and runs one unit per SM: a single long sequence (131 072 tokens, 16 heads)
// then occupies 16 SMs.  The prep has every (chunk, head) as independent work for every SM, and
// the sweep's serial chain per chunk is only U = T_b V - W S, O, and the state update (SGLang PR
// 34820 page: the per-chunk state loop of the Helion listing is the only serial part; "state
// semantics" page, section 5: TP does not shorten that chain).  The cost is the workspace round
// trip of the operands (about 2 KiB per token-head each way).
//
// One long sequence with few heads leaves most SMs idle in the sweep while the prep has long
// finished.  Across a chunk the state map is affine, S' = M S + K~^T U~ with M = Diag(e^{G_63})
// - K~^T W, so with few enough heads the chunks are cut into segments swept at the same time:
// each middle segment's matrix product Phi and offset B, the segment start states chained from
// them (S_{s+1} = Phi_s S_s + B_s), then every segment swept from its start.  With more heads
// the segments run one after another instead, each segment's sweep beside the prep of the next
// in one launch (the halves share no data and never wait on each other), with the state handed
// from segment to segment through the workspace, exactly.
//
// Inputs may be bf16 or fp32: the prep reads fp32 q, k and the raw gate from global memory and
// splits its products as for bf16; the sweep splits fp32 V into bf16 hi/lo tiles itself.
//
// Precision is the single-pass kernel's: operands that are not exact bf16 inputs are split into
// bf16 hi + lo, products hi*hi + hi*lo + lo*hi, state fp32 in TMEM.  A chunk whose decay factors
// leave the range of that form (a half chunk's product of 1/alpha above 2^64) is flagged by the
// prep and evaluated token by token by the sweep, exactly in fp32.
#include <string.h>

#include "kda_common.cuh"
#include "kda_host.h"
#include "prefill.h"
#include "umma.cuh"

namespace kda {
namespace {

using namespace umma;

constexpr int kThreads = 512;  // 16 warps: four per TMEM lane quarter
constexpr int kTrack2p = 512;  // snapshot requests per sequence

// ---- one operand block per (chunk, head): the sweep's shared-memory image
constexpr uint32_t OP_QW = 0;         // [QG; -W hi; -W lo]  B, MN-major, 3 x 16 KiB
constexpr uint32_t OP_TB = 49152;     // [T_b hi; T_b lo]    B, K-major, 128 rows
constexpr uint32_t OP_GAM = 65536;    // e^{G_63}, fp32 [128]; +512: int32 flag (1 = token path)
constexpr uint32_t OP_QGLO = 66560;   // QG lo (fp32 outputs), MN-major
constexpr uint32_t OP_KTP = 82944;    // [KT hi; P]          B, K-major, 192 rows
constexpr uint32_t OP_PLO = 107520;   // P lo (fp32 outputs), K-major, 64 rows
constexpr uint32_t OP_KTLO = 115712;  // KT lo, K-major, 128 rows
constexpr uint32_t OP_BYTES = 132096;
constexpr uint32_t OP_FLAG = OP_GAM + 512;
// part A ([0, .)) feeds the U / O products; part B ([OP_KTP, OP_BYTES)) the state update, in
// one piece for fp32 outputs and without P lo (two pieces) for bf16 outputs
constexpr uint32_t opa_bytes(bool bf16_out) { return bf16_out ? 66560u : 82944u; }
constexpr uint32_t OPB1_BYTES_BF16 = OP_PLO - OP_KTP;     // [KT hi; P]
constexpr uint32_t OPB2_BYTES_BF16 = OP_BYTES - OP_KTLO;  // KT lo
constexpr uint32_t opb_bytes(bool bf16_out) { return bf16_out ? OPB1_BYTES_BF16 + OPB2_BYTES_BF16 : OP_BYTES - OP_KTP; }

// ---- plan area at the head of the workspace
constexpr size_t PL_ORDER = 0;         // [kMaxOrderN] sequences, longest first
constexpr size_t PL_BASE = 16384;      // [N + 1] first chunk of each sequence
constexpr size_t PL_META = 33280;      // [0]: chunks in all
constexpr size_t PL_SOC = 33536;       // [n_max] sequence of each chunk
constexpr int kPlanThreads = 1024;

int64_t max_chunks(int32_t T_tot, int32_t N) { return ((int64_t)T_tot + 63 * (int64_t)N) / kChunk; }
// [n_max] int2 (first token row, length) of each chunk, after the sequence table
__host__ __device__ constexpr size_t cinfo_offset(int64_t n_max) { return (PL_SOC + (size_t)n_max * 4 + 15) & ~(size_t)15; }
size_t ops_offset(int64_t n_max) { return (cinfo_offset(n_max) + (size_t)n_max * 8 + 1023) & ~(size_t)1023; }

constexpr uint32_t kWaitLimit = 1u << 18;    // polls of ~4 us (try_wait suspends): ~1 s
constexpr float kFactorMax = 1.8446744e19f;  // 2^64

__device__ __forceinline__ float bf16_at(const uint8_t* sm, uint32_t off) {
    return __uint_as_float((uint32_t)(*reinterpret_cast<const uint16_t*>(sm + off)) << 16);
}

__device__ __forceinline__ void st16(uint8_t* sm, uint32_t off, uint4 v) {
    *reinterpret_cast<uint4*>(sm + off) = v;
}

// Smallest snapshot request above chunk j (INT_MAX if none): the state pass tests one index per
// chunk instead of walking all M requests.
__device__ __forceinline__ int next_tracked(const int* s_trk, int M, int j) {
    int best = 0x7fffffff;
    for (int m = 0; m < M; ++m) {
        const int jj = s_trk[m];
        if (jj > j && jj < best) best = jj;
    }
    return best;
}

// ----------------------------------------------------------------------------
// plan: chunk counts, their prefix sums, the sequence of every chunk, longest-first order

__global__ void __launch_bounds__(kPlanThreads) prefill_plan_kernel(const int32_t* __restrict__ cu, int N,
                                                                     int T_tot, int64_t n_max,
                                                                     int32_t* __restrict__ plan) {
    __shared__ int s_cnt[kMaxOrderN];
    __shared__ int s_warp[kPlanThreads / 32];
    int32_t* order = plan + PL_ORDER / 4;
    int32_t* base = plan + PL_BASE / 4;
    int32_t* meta = plan + PL_META / 4;
    int32_t* soc = plan + PL_SOC / 4;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    for (int n = tid; n < kMaxOrderN; n += kPlanThreads) {
        int cnt = 0;
        if (n < N) {
            const int t0 = cu[n], t1 = cu[n + 1];
            const bool ok = t0 >= 0 && t1 >= t0 && t1 <= T_tot && (n > 0 || t0 == 0);
            cnt = ok ? (t1 - t0 + kChunk - 1) / kChunk : 0;  // a malformed sequence: no chunks
        }
        s_cnt[n] = cnt;
    }
    __syncthreads();
    // exclusive prefix sum; thread tid owns sequences 4 tid .. 4 tid + 3
    int loc[4], run = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        loc[e] = run;
        run += s_cnt[4 * tid + e];
    }
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        const int w = s_warp[lane];
        int iw = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, iw, o);
            if (lane >= o) iw += y;
        }
        s_warp[lane] = iw - w;
    }
    __syncthreads();
    const int excl = s_warp[wid] + incl - run;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int n = 4 * tid + e;
        if (n <= N) base[n] = excl + loc[e];
    }
    if (tid == kPlanThreads - 1) meta[0] = excl + run;  // every sequence is counted by here
    __syncthreads();
    // the sequence, first row and length of every chunk (one thread per sequence), and the
    // order: most chunks first
    int2* cinfo = reinterpret_cast<int2*>(reinterpret_cast<uint8_t*>(plan) + cinfo_offset(n_max));
    for (int n = tid; n < N; n += kPlanThreads) {
        const int b = base[n], cnt = s_cnt[n];
        const int t0 = cnt > 0 ? cu[n] : 0, L = cnt > 0 ? cu[n + 1] - t0 : 0;
        for (int jj = 0; jj < cnt && (int64_t)b + jj < n_max; ++jj) {
            soc[b + jj] = n;
            cinfo[b + jj] = make_int2(t0 + jj * kChunk, min(kChunk, L - jj * kChunk));
        }
        int rank = 0;
        for (int m = 0; m < N; ++m) rank += (s_cnt[m] > cnt) || (s_cnt[m] == cnt && m < n);
        order[rank] = n;
    }
}

// ----------------------------------------------------------------------------
// prep: the state-independent half of every (chunk, head)
//
// Persistent: each CTA walks (chunk, head) items blockIdx.x, + gridDim.x, ...  Per item:
//   gate pass -> L/R -> MMA 1 ([A; P]) issued; K_G / Q_G / K~ built while it runs ->
//   A/P extraction -> triangular solve -> T_b -> MMA 2 (W) -> W extraction -> bulk store
// The next item's raw gate tile is requested right after this item's gate pass and its q / k
// tiles after the K_G pass (each tile as soon as this item's copy is consumed); the image leaves
// by asynchronous bulk stores that the next item waits on only before its L/R stores.

// shared memory (bytes from a 1024-aligned base)
constexpr uint32_t PR_RAW = 0;  // raw q, k, g tiles, row-major bf16 [t][128]
constexpr uint32_t PR_Q = PR_RAW, PR_K = PR_RAW + 16384, PR_G = PR_RAW + 32768;
constexpr uint32_t PR_IMG = 49152;             // the operand block image
constexpr uint32_t PR_EXT = PR_IMG + OP_BYTES;  // 32 KiB beside it
// MMA 1's operands live only in regions written after MMA 1 has read them (the W tiles, the
// T_b tile, P and P lo) and in PR_EXT, so K_G / Q_G / K~, e^{G_63} and the flag (early regions)
// can be written while MMA 1 runs.  The solve's scratch follows MMA 1 the same way.
constexpr uint32_t PR_L_HI = PR_IMG + OP_QW + 16384;  // L hi (A, MN-major, 32 KiB): the W tiles
constexpr uint32_t PR_L_LO = PR_EXT;                  // L lo
constexpr uint32_t PR_R_HI = PR_IMG + OP_TB;          // R hi (B, MN-major, 16 KiB): the T_b tile
constexpr uint32_t PR_R_LO = PR_IMG + OP_KTP + 16384; // R lo: P and P lo
constexpr uint32_t PR_R_LBO = PR_R_LO - PR_R_HI;      // [R hi; R lo] as one N = 128 operand
constexpr uint32_t PR_N = PR_IMG + OP_QW + 16384;     // N^T fp32 [64][68] (after MMA 1)
constexpr uint32_t PR_T = PR_EXT, PR_Y1 = PR_EXT + 17408, PR_Y2 = PR_EXT + 19968;
constexpr uint32_t PR_MISC = PR_EXT + 32768;
constexpr uint32_t PR_SMEM = PR_MISC + 5120 + 1024;
constexpr int NLD = 68;  // fp32 row stride of the N / T matrices
static_assert(PR_L_HI + 32768 <= PR_IMG + OP_TB, "L hi must stay inside the W tiles");
static_assert(PR_R_LO + 16384 <= PR_IMG + OP_KTLO, "R lo must stay inside P and P lo");
static_assert(PR_N + 64 * NLD * 4 <= PR_IMG + OP_TB, "N^T must stay inside the W tiles");
static_assert(PR_Y2 + 32 * 36 * 4 <= PR_EXT + 32768, "solve scratch exceeds its region");
static_assert(PR_SMEM <= 232448, "prep shared memory plan exceeds the per-CTA limit");

// TMEM (256 columns): [A;P] accumulator (hi-R | lo-R parts), W^T, KG hi/lo A operand
constexpr uint32_t PT_AP = 0, PT_W = 128, PT_KG_HI = 192, PT_KG_LO = 224, PT_COLS = 256;

// The prep's 512 threads synchronise on barrier 1 with an explicit count, so that a CTA of a
// wider launch (the pipelined long-sequence path) can run it while its other warps exit.
constexpr int kPrepBar = 1;

// The items of chunks [c_begin, c_end) (global chunk index), walked by CTA `cta` of `ncta`.
template <bool kBf16Out, bool kF32In>
__device__ __forceinline__ void prep_body(const CUtensorMap* qmap, const CUtensorMap* kmap,
                                          const CUtensorMap* gmap, const PrefillArgs& p,
                                          const int32_t* __restrict__ plan, int64_t n_max,
                                          uint8_t* __restrict__ ops, int cta, int ncta, int64_t c_begin,
                                          int64_t c_end) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(sm);
    const uint32_t sb4 = sb >> 4;
    float* s_beta = reinterpret_cast<float*>(sm + PR_MISC);  // 64
    float* s_nk = s_beta + 64;                               // 64: L2 factors of the key rows
    float* s_nq = s_nk + 64;                                 // 64: of the query rows (x scale)
    float* s_seg_a = s_nq + 64;                              // [4][128]: prod of alpha per token quarter
    float* s_seg_i = s_seg_a + 512;                          // [4][128]: prod of 1/alpha per quarter
    uint64_t* s_mbar = reinterpret_cast<uint64_t*>(s_seg_i + 512);  // MMA, raw q / k tiles, raw gate tile
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(s_mbar + 3);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quarter = warp & 3;  // TMEM lane quarter this warp may access
    const int cq = warp >> 2;      // column quarter this warp takes in TMEM passes
    const int row = quarter * 32 + lane;
    const int ci = tid & 127, tq = tid >> 7;  // channel passes: key channel, token quarter
    const bool store_lane = lane == 0 && warp >= 7 && warp <= 9;  // issue the image's bulk stores
    const int H = p.H;
    const int64_t n_chunks_all = min((int64_t)plan[PL_META / 4], n_max);
    const int64_t w_lo = c_begin * H;                          // this call's first item
    const int64_t items = min(n_chunks_all, c_end) * H;        // one past its last
    if (w_lo + cta >= items) return;
    const bool l2 = (p.flags & KDA_QK_L2NORM) != 0;

    if (warp == 0) tmem_alloc(smem_u32(s_tmem), PT_COLS);
    if (tid == 0) {
        mbar_init(smem_u32(s_mbar), 1);
        mbar_init(smem_u32(s_mbar + 1), 1);
        mbar_init(smem_u32(s_mbar + 2), 1);
    }
    fence_before();
    bar_named(kPrepBar, kThreads);
    fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t mbar = smem_u32(s_mbar), mbar_qk = smem_u32(s_mbar + 1), mbar_g = smem_u32(s_mbar + 2);
    uint32_t phase = 0, phase_qk = 0, phase_g = 0;
    // raw-tile copies issued and not yet waited on (every thread tracks them)
    bool qk_pending = false, g_pending = false;
    bool timed_out = false;

    struct Item {
        int64_t c;
        int h, c0, Lc;
    };
    const int2* cinfo = reinterpret_cast<const int2*>(reinterpret_cast<const uint8_t*>(plan) + cinfo_offset(n_max));
    auto item_at = [&](int64_t c, int hh) {  // one 8-byte load
        Item it;
        it.c = c;
        it.h = hh;
        const int2 ci2 = cinfo[c];
        it.c0 = ci2.x;
        it.Lc = ci2.y;
        return it;
    };
    // item w is (chunk w / H, head w % H); consecutive items of this CTA are ncta apart
    const int64_t step_c = ncta / H;
    const int step_h = (int)(ncta - step_c * H);
    // raw tiles of an item (bf16: 128-channel x 64-token tensor-map boxes; rows past the
    // sequence are cleared once they land).  The gate tile is read by the gate pass only, so the
    // next item's is requested right after it; the q and k tiles are read until the K_G pass and
    // wait for it, together with the item's raw beta bits.  Called by every thread once every
    // thread is past its reads of the tiles concerned.
    auto prefetch_g = [&](const Item& it) {
        if constexpr (!kF32In) {
            if (lane == 0 && warp == 3) {
                fence_async_smem();
                mbar_expect_tx(mbar_g, 16384u);
                tma_load_2d(sb + PR_G, gmap, it.h * kD, it.c0, mbar_g);
            }
            g_pending = true;
        }
    };
    auto prefetch_qk = [&](const Item& it, uint32_t& beta_bits) {
        if constexpr (!kF32In) {
            // one copy per issuing thread, in two warps (a copy that lands before the expected
            // byte count is posted only takes the count below zero while the arrival is pending)
            if (lane == 0 && (warp == 1 || warp == 2)) {
                fence_async_smem();
                if (warp == 1) mbar_expect_tx(mbar_qk, 2u * 16384u);
                tma_load_2d(sb + (warp == 1 ? PR_Q : PR_K), warp == 1 ? qmap : kmap, it.h * kD, it.c0, mbar_qk);
            }
            qk_pending = true;
        }
        if (tid < 64) {
            const size_t bi = (size_t)(it.c0 + min(tid, it.Lc - 1)) * H + it.h;
            if constexpr (kF32In)
                beta_bits = __float_as_uint(__ldg(static_cast<const float*>(p.beta_raw) + bi));
            else
                beta_bits = __ldg(static_cast<const unsigned short*>(p.beta_raw) + bi);
        }
    };

    uint32_t beta_bits = 0;
    Item cur = item_at((w_lo + cta) / H, (int)((w_lo + cta) % H));
    // the item ncta after `it`, or `it` again when there is none: the choice is made on the
    // indices, so that the 8-byte load is always in range and nothing waits on it until the
    // item's fields are used (a choice between loaded values stalled every thread at the top of
    // each item for the load's full latency)
    auto next_or_same = [&](const Item& it, bool exists) {
        int64_t c2 = it.c;
        int h2 = it.h;
        if (exists) {
            c2 += step_c;
            h2 += step_h;
            if (h2 >= H) {
                h2 -= H;
                ++c2;
            }
        }
        return item_at(c2, h2);
    };
    // raw element (t, ci) of the current item: bf16 from its staged tile, fp32 activations
    // straight from global memory (rows past the sequence read as 0 either way)
    auto raw_at = [&](const void* g32, uint32_t tile, int t) -> float {
        if constexpr (kF32In) {
            return t < cur.Lc ? __ldg(static_cast<const float*>(g32) + ((size_t)(cur.c0 + t) * H + cur.h) * kD + ci)
                              : 0.f;
        } else {
            return bf16_at(sm, tile + t * 256 + ci * 2);
        }
    };
    // key / query element (t, ci) as the recurrence uses it (q also times scale)
    auto key_at = [&](int t) {
        const float x = raw_at(p.k, PR_K, t);
        return l2 ? x * s_nk[t] : x;
    };
    auto query_at = [&](int t) {
        const float x = raw_at(p.q, PR_Q, t);
        return l2 ? x * s_nq[t] : x * p.scale;
    };
    prefetch_g(cur);
    prefetch_qk(cur, beta_bits);
    for (int64_t w = w_lo + cta; w < items; w += ncta) {
        const int64_t w_next = w + ncta;
        const bool has_next = w_next < items;
        const bool has_next2 = w_next + ncta < items;
        const Item nxt = next_or_same(cur, has_next);
        // the item after it, for the L2 prefetch: its 8-byte load is issued here, used much later
        const Item nxt2 = next_or_same(nxt, has_next2);
        const int Lc = cur.Lc, h = cur.h;
        uint8_t* blk = ops + ((size_t)cur.c * H + h) * OP_BYTES;

        // the gate tile (a timed-out wait is decided at the gate pass's barrier; rows past the
        // sequence are read but their decays replaced by 1)
        bool okg = true;
        if constexpr (!kF32In) {
            okg = mbar_wait(mbar_g, phase_g, kWaitLimit);
            phase_g ^= 1;
            g_pending = false;
        }
        // beta is first read after the channel pass's barrier
        if (tid < 64) {
            const float braw = __uint_as_float(kF32In ? beta_bits : beta_bits << 16);
            s_beta[tid] = tid < Lc ? beta_act(braw, p.flags) : 0.f;
        }

        // ---- channel pass: this thread's channel ci over tokens 16*tq .. 16*tq+15
        float al[16], iv[16];
        float m_big = 1.f;  // product of the factors >= 1 this quarter contributes to its half
        {
            with_gate_form(p.flags, [&](uint32_t form) {
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int t = 16 * tq + u;
                    const Decay dc = decay_of(raw_at(p.gate_raw, PR_G, t), form);
                    al[u] = t < Lc ? dc.a : 1.f;
                    iv[u] = t < Lc ? dc.inv : 1.f;
                }
            });
            float pa = 1.f, pi = 1.f;
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                pa *= al[u];
                pi *= iv[u];
                if (tq != 0 || u > 0) m_big *= iv[u];
            }
            s_seg_a[tq * 128 + ci] = pa;
            s_seg_i[tq * 128 + ci] = pi;
        }
        if (bar_named_or(kPrepBar, kThreads, !okg)) {
            timed_out = true;
            break;
        }
        // every gate read of this item is done: the next item's gate tile may land
        if (has_next) prefetch_g(nxt);
        bool bad = false;
        // largest factor a half uses: prod of 1/alpha over (0, 31] (half 0) or [32, 63] (half 1)
        if (tq == 0) bad = !(m_big * s_seg_i[128 + ci] <= kFactorMax);
        if (tq == 2) bad = !(m_big * s_seg_i[384 + ci] <= kFactorMax);
        // the q and k tiles (a timed-out wait is decided at the barrier after the L/R arithmetic)
        bool okqk = true;
        if constexpr (!kF32In) {
            okqk = mbar_wait(mbar_qk, phase_qk, kWaitLimit);
            phase_qk ^= 1;
            qk_pending = false;
            if (Lc < kChunk) {
                // rows past the sequence (the next one's, or zero-filled past T_tot) -> 0, so that
                // no other row's values (possibly non-finite) enter this chunk
                for (int e = tid; e < 2 * 64 * 16; e += kThreads) {
                    const int t = (e >> 4) & 63, ch = e & 15;
                    if (t >= Lc) st16(sm, (e >> 10 ? PR_K : PR_Q) + t * 256 + ch * 16, make_uint4(0, 0, 0, 0));
                }
                bar_named(kPrepBar, kThreads);
            }
        }
        if (l2) {
            // KDA_QK_L2NORM: factors of the key and query rows, a warp per 4 rows
#pragma unroll
            for (int tt = 0; tt < 4; ++tt) {
                const int t = 4 * warp + tt;
                float4 kx, qx;
                if constexpr (kF32In) {
                    kx = qx = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (t < Lc) {
                        const size_t e = ((size_t)(cur.c0 + t) * H + h) * kD + lane * 4;
                        kx = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.k) + e));
                        qx = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(p.q) + e));
                    }
                } else {
                    kx = State<kStateBF16>::widen(*reinterpret_cast<const uint2*>(sm + PR_K + t * 256 + lane * 8));
                    qx = State<kStateBF16>::widen(*reinterpret_cast<const uint2*>(sm + PR_Q + t * 256 + lane * 8));
                }
                float sk = f4_dot(kx, kx), sq = f4_dot(qx, qx);
                warp_sum2(sk, sq);
                if (lane == 0) {
                    s_nk[t] = l2norm_factor(sk);
                    s_nq[t] = l2norm_factor(sq) * p.scale;
                }
            }
            bar_named(kPrepBar, kThreads);
        }

        // ---- L = [k; q] e^{G_t - G_31}, R = k e^{G_31 - G_s}: quarters 0, 1 backward
        //      from token 31, quarters 2, 3 forward from token 32.  L lo goes to shared memory at
        //      once (no image store reads its region); L hi and R, whose tiles alias the image's
        //      W, T_b and P tiles, wait in registers until the previous item's image stores have
        //      read those tiles, so that the wait overlaps this arithmetic.
        uint4 lkh[2], lqh[2], rh[2], rl[2];
        auto lr_split = [&](int g8, float(&lk)[8], float(&lq)[8], float(&r)[8]) {
            const int tt = 16 * tq + g8 * 8;
            uint4 lo;
            split8p(lk, lkh[g8], lo);
            st16(sm, PR_L_LO + chunk_mn(tt, ci, 1024, 2048), lo);
            split8p(lq, lqh[g8], lo);
            st16(sm, PR_L_LO + chunk_mn(64 + tt, ci, 1024, 2048), lo);
            split8p(r, rh[g8], rl[g8]);
        };
        if (tq < 2) {
            float sa = 1.f, si = 1.f;  // prod over (u, 31] of alpha and of 1/alpha
            if (tq == 0) {
                sa = s_seg_a[128 + ci];
                si = s_seg_i[128 + ci];
            }
#pragma unroll
            for (int g8 = 1; g8 >= 0; --g8) {
                float lk[8], lq[8], r[8];
#pragma unroll
                for (int w8 = 7; w8 >= 0; --w8) {
                    const int u = g8 * 8 + w8, t = 16 * tq + u;
                    const float kk = key_at(t);
                    const float qq = query_at(t);
                    lk[w8] = kk * si;
                    lq[w8] = qq * si;
                    r[w8] = kk * sa;
                    sa *= al[u];
                    si *= iv[u];
                }
                lr_split(g8, lk, lq, r);
            }
        } else {
            float fa = 1.f, fi = 1.f;  // prod over [32, t] of alpha and of 1/alpha
            if (tq == 3) {
                fa = s_seg_a[256 + ci];
                fi = s_seg_i[256 + ci];
            }
#pragma unroll
            for (int g8 = 0; g8 < 2; ++g8) {
                float lk[8], lq[8], r[8];
#pragma unroll
                for (int w8 = 0; w8 < 8; ++w8) {
                    const int u = g8 * 8 + w8, t = 16 * tq + u;
                    const float kk = key_at(t);
                    const float qq = query_at(t);
                    fa *= al[u];
                    fi *= iv[u];
                    lk[w8] = kk * fa;
                    lq[w8] = qq * fa;
                    r[w8] = kk * fi;
                }
                lr_split(g8, lk, lq, r);
            }
        }
        if (store_lane) bulk_wait_read_all();  // the previous item's image has left shared memory
        if (bar_named_or(kPrepBar, kThreads, bad || !okqk)) {
            if (bar_named_or(kPrepBar, kThreads, !okqk)) {
                timed_out = true;
                break;
            }
            // the sweep evaluates this chunk token by token from the raw inputs
            if (tid == 0) *reinterpret_cast<int32_t*>(blk + OP_FLAG) = 1;
            if (has_next) prefetch_qk(nxt, beta_bits);  // every thread is past its raw reads
            cur = nxt;
            continue;
        }
#pragma unroll
        for (int g8 = 0; g8 < 2; ++g8) {
            const int tt = 16 * tq + g8 * 8;
            st16(sm, PR_L_HI + chunk_mn(tt, ci, 1024, 2048), lkh[g8]);
            st16(sm, PR_L_HI + chunk_mn(64 + tt, ci, 1024, 2048), lqh[g8]);
            st16(sm, PR_R_HI + chunk_mn(tt, ci, 1024, 1024), rh[g8]);
            st16(sm, PR_R_LO + chunk_mn(tt, ci, 1024, 1024), rl[g8]);
        }
        fence_async_smem();
        fence_before();
        bar_named(kPrepBar, kThreads);
        fence_after();
        // ---- MMA 1: [A; P] = [L_k; L_q] R^T: L_hi [R_hi; R_lo]^T (N = 128) + L_lo R_hi^T
        if (tid == 0) {
            const uint32_t id2 = idesc_bf16(128, 128, true, true, false);
            const uint32_t id1 = idesc_bf16(128, 64, true, true, false);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma(tmem + PT_AP, desc_mn4(sb4 + PR_L_HI / 16, 1024, 2048, s),
                    desc_mn4(sb4 + PR_R_HI / 16, PR_R_LBO, 1024, s), id2, s != 0);
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma(tmem + PT_AP, desc_mn4(sb4 + PR_L_LO / 16, 1024, 2048, s),
                    desc_mn4(sb4 + PR_R_HI / 16, PR_R_LBO, 1024, s), id1, 1u);
            commit(mbar);
        }
        // ---- while MMA 1 runs: KG = k e^{G} (A, [i][s], TMEM), QG = q e^{G} (B, MN-major),
        //      KT = k e^{G_63 - G} (B, K-major), e^{G_63} and the flag word
        {
            const float a0 = s_seg_a[ci], a1 = s_seg_a[128 + ci], a2 = s_seg_a[256 + ci],
                        a3 = s_seg_a[384 + ci];
            // e^{G_t}: running product from the chunk start; e^{G_63 - G_t}: product over (t, 63]
            float fw = tq == 0 ? 1.f : tq == 1 ? a0 : tq == 2 ? a0 * a1 : (a0 * a1) * a2;
            float bw = tq == 3 ? 1.f : tq == 2 ? a3 : tq == 1 ? a2 * a3 : a1 * (a2 * a3);
            if (tq == 0) reinterpret_cast<float*>(sm + PR_IMG + OP_GAM)[ci] = (a0 * a1) * (a2 * a3);
            if (tid == 0) *reinterpret_cast<int32_t*>(sm + PR_IMG + OP_FLAG) = 0;
            uint32_t kgh[8], kgl[8];  // KG row ci, tokens 16*tq.., packed bf16 pairs
#pragma unroll
            for (int c8 = 0; c8 < 2; ++c8) {
                float kg[8], qg[8];
#pragma unroll
                for (int w8 = 0; w8 < 8; ++w8) {
                    const int u = 8 * c8 + w8, t = 16 * tq + u;
                    fw *= al[u];
                    kg[w8] = key_at(t) * fw;
                    qg[w8] = query_at(t) * fw;
                }
                const int s0 = 16 * tq + 8 * c8;
                uint4 hi, lo;
                split8p(kg, hi, lo);
                kgh[4 * c8] = hi.x; kgh[4 * c8 + 1] = hi.y; kgh[4 * c8 + 2] = hi.z; kgh[4 * c8 + 3] = hi.w;
                kgl[4 * c8] = lo.x; kgl[4 * c8 + 1] = lo.y; kgl[4 * c8 + 2] = lo.z; kgl[4 * c8 + 3] = lo.w;
                if constexpr (kBf16Out) {
                    st16(sm, PR_IMG + OP_QW + chunk_mn(s0, ci, 1024, 1024), pack8(qg));
                } else {
                    split8p(qg, hi, lo);
                    st16(sm, PR_IMG + OP_QW + chunk_mn(s0, ci, 1024, 1024), hi);
                    st16(sm, PR_IMG + OP_QGLO + chunk_mn(s0, ci, 1024, 1024), lo);
                }
            }
#pragma unroll
            for (int c8 = 1; c8 >= 0; --c8) {
                float kt[8];
#pragma unroll
                for (int w8 = 7; w8 >= 0; --w8) {
                    const int u = 8 * c8 + w8, t = 16 * tq + u;
                    kt[w8] = key_at(t) * bw;
                    bw *= al[u];
                }
                const int s0 = 16 * tq + 8 * c8;
                uint4 hi, lo;
                split8p(kt, hi, lo);
                st16(sm, PR_IMG + OP_KTP + chunk_k(ci, s0, 128), hi);
                st16(sm, PR_IMG + OP_KTLO + chunk_k(ci, s0, 128), lo);
            }
            st8u(tl + PT_KG_HI + tq * 8, kgh);  // lane ci of this warp's quarter
            st8u(tl + PT_KG_LO + tq * 8, kgl);
            wait_st();
        }
        {
            const bool ok1 = mbar_wait(mbar, phase, kWaitLimit);
            phase ^= 1;
            fence_after();
            if (bar_named_or(kPrepBar, kThreads, !ok1)) {
                timed_out = true;
                break;
            }
        }
        // every q / k read of this item is done: the next item's tiles may land, and the item
        // after it is pulled into L2
        if (has_next) prefetch_qk(nxt, beta_bits);
        if constexpr (!kF32In) {
            if (lane == 0 && warp >= 4 && warp <= 6 && has_next2)
                tma_prefetch_2d(warp == 4 ? qmap : warp == 5 ? kmap : gmap, nxt2.h * kD, nxt2.c0);
        }

        // ---- A -> N = Diag(beta) A (strict lower, stored transposed: Nt[s][t] = N[t][s]),
        //      P -> bf16 operand (lower incl. diagonal)
        {
            float v[16], v2[16];
            ld16(tl + PT_AP + cq * 16, v);
            ld16(tl + PT_AP + 64 + cq * 16, v2);
#pragma unroll
            for (int q = 0; q < 16; ++q) v[q] += v2[q];
            float* Nt = reinterpret_cast<float*>(sm + PR_N);
            if (quarter < 2) {
                const int t = row;
                const float bt = s_beta[t];
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const int s = cq * 16 + q;
                    Nt[s * NLD + t] = s < t ? bt * v[q] : 0.f;
                }
            } else {
                const int t = row - 64;
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    const int s = cq * 16 + q;
                    if (s > t) v[q] = 0.f;
                }
#pragma unroll
                for (int c8 = 0; c8 < 2; ++c8) {
                    if constexpr (kBf16Out) {
                        st16(sm, PR_IMG + OP_KTP + 16384 + chunk_k(t, cq * 16 + 8 * c8, 64), pack8(v + 8 * c8));
                    } else {
                        uint4 hi, lo;
                        split8p(v + 8 * c8, hi, lo);
                        st16(sm, PR_IMG + OP_KTP + 16384 + chunk_k(t, cq * 16 + 8 * c8, 64), hi);
                        st16(sm, PR_IMG + OP_PLO + chunk_k(t, cq * 16 + 8 * c8, 64), lo);
                    }
                }
            }
        }
        bar_named(kPrepBar, kThreads);
        // ---- T = (I + N)^-1 (unit lower triangular): 16x16 diagonal blocks by forward
        //      substitution, then the off-diagonal blocks by block substitution, level by level
        //      (16 -> 32 -> 64).  The level products split their sums over 2-4 threads (shuffle
        //      reductions), and the last one writes T_b = T Diag(beta) as the bf16 hi/lo operand.
        //      Only entries on or below the diagonal of T are read: the 16x16 blocks above the
        //      diagonal are never written.
        {
            const float* Nt = reinterpret_cast<const float*>(sm + PR_N);
            float* Tm = reinterpret_cast<float*>(sm + PR_T);
            if (tid < 64) {
                // column jc of the inverse of diagonal block b: x = e_jc, then for each s
                // (final from here on) x[r] -= N[r][s] x[s] for r > s
                const int b = tid >> 4, jc = tid & 15, o = 16 * b;
                float x[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) x[r] = (r == jc) ? 1.f : 0.f;
#pragma unroll
                for (int s = 0; s < 15; ++s) {
                    float nr[16];
#pragma unroll
                    for (int r4 = (s + 1) / 4; r4 < 4; ++r4) {
                        const float4 n4 = *reinterpret_cast<const float4*>(&Nt[(o + s) * NLD + o + 4 * r4]);
                        nr[4 * r4] = n4.x;
                        nr[4 * r4 + 1] = n4.y;
                        nr[4 * r4 + 2] = n4.z;
                        nr[4 * r4 + 3] = n4.w;
                    }
                    const float xs = x[s];
#pragma unroll
                    for (int r = s + 1; r < 16; ++r) x[r] = fmaf(-nr[r], xs, x[r]);
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) Tm[(o + r) * NLD + o + jc] = x[r];
            }
            bar_named(kPrepBar, kThreads);
            // level 1: T[a][a-1] = -T_aa N[a][a-1] T_{a-1,a-1}, a in {1, 3}; a thread owns
            // row r and 4 adjacent columns of one 16x16 block
            float* Y1 = reinterpret_cast<float*>(sm + PR_Y1);  // [2][16][20]
            const int w1 = tid >> 6, r1 = (tid & 63) >> 2, c1 = (tid & 3) * 4;
            const int oa = 32 * w1 + 16, ob = 32 * w1;
            if (tid < 128) {
                float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const float nv = Nt[(ob + u) * NLD + oa + r1];
                    const float4 tv = *reinterpret_cast<const float4*>(&Tm[(ob + u) * NLD + ob + c1]);
                    y.x = fmaf(nv, tv.x, y.x);
                    y.y = fmaf(nv, tv.y, y.y);
                    y.z = fmaf(nv, tv.z, y.z);
                    y.w = fmaf(nv, tv.w, y.w);
                }
                *reinterpret_cast<float4*>(&Y1[(w1 * 16 + r1) * 20 + c1]) = y;
            }
            bar_named(kPrepBar, kThreads);
            if (tid < 128) {
                // T_aa is lower triangular: terms s > r1 are zero (and read as zero)
                float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int s2 = 0; s2 < 16; ++s2) {
                    const float tv = Tm[(oa + r1) * NLD + oa + s2];
                    const float4 yv = *reinterpret_cast<const float4*>(&Y1[(w1 * 16 + s2) * 20 + c1]);
                    z.x = fmaf(tv, yv.x, z.x);
                    z.y = fmaf(tv, yv.y, z.y);
                    z.z = fmaf(tv, yv.z, z.z);
                    z.w = fmaf(tv, yv.w, z.w);
                }
                *reinterpret_cast<float4*>(&Tm[(oa + r1) * NLD + ob + c1]) = make_float4(-z.x, -z.y, -z.z, -z.w);
            }
            bar_named(kPrepBar, kThreads);
            // level 2, first product: Y2 = N[32:64, 0:32] T[0:32, 0:32].  Warp = (4-column group
            // c2, half of the rows); lane = (row, parity of the sum), the parities meet by shuffle.
            // T[u][c] is zero for u < c, so the sum starts at c2.
            float* Y2 = reinterpret_cast<float*>(sm + PR_Y2);  // [32][36]
            {
                const int c2 = 4 * (warp & 7), r2 = 16 * (warp >> 3) + (lane & 15), par = lane >> 4;
                float4 y = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
                for (int u = c2 + par; u < 32; u += 2) {
                    const float nv = Nt[u * NLD + 32 + r2];
                    const float4 tv = *reinterpret_cast<const float4*>(&Tm[u * NLD + c2]);
                    y.x = fmaf(nv, tv.x, y.x);
                    y.y = fmaf(nv, tv.y, y.y);
                    y.z = fmaf(nv, tv.z, y.z);
                    y.w = fmaf(nv, tv.w, y.w);
                }
                y.x += __shfl_xor_sync(0xffffffffu, y.x, 16);
                y.y += __shfl_xor_sync(0xffffffffu, y.y, 16);
                y.z += __shfl_xor_sync(0xffffffffu, y.z, 16);
                y.w += __shfl_xor_sync(0xffffffffu, y.w, 16);
                if (par == 0) *reinterpret_cast<float4*>(&Y2[r2 * 36 + c2]) = y;
            }
            bar_named(kPrepBar, kThreads);
            // level 2, second product, and T_b = T Diag(beta) -> bf16 hi/lo operand [t][s].
            // Thread = (row pair t_lo / 32 + t_lo, column quad c4 of 16).  Rows 0-31 and the
            // quads right of column 32 are copies of T (zero above the diagonal); the quads
            // of T[32:64, 0:32] = -T[32:64, 32:64] Y2 split their sum between lanes c4 and
            // c4 + 8 (even / odd terms).
            {
                const int c4 = tid & 15, t_lo = tid >> 4;
                auto emit = [&](int t, float4 x) {
                    const int s0 = 4 * c4;
                    x.x *= s_beta[s0];
                    x.y *= s_beta[s0 + 1];
                    x.z *= s_beta[s0 + 2];
                    x.w *= s_beta[s0 + 3];
                    uint2 hi, lo;
                    split2p(x.x, x.y, hi.x, lo.x);
                    split2p(x.z, x.w, hi.y, lo.y);
                    const uint32_t off = PR_IMG + OP_TB + chunk_k(t, s0 & ~7, 64) + (s0 & 4) * 2;
                    *reinterpret_cast<uint2*>(sm + off) = hi;
                    *reinterpret_cast<uint2*>(sm + off + 8192) = lo;
                };
                auto copy_of = [&](int t) {  // T[t][4 c4 .. 4 c4 + 3], zero above the diagonal
                    const int s0 = 4 * c4;
                    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (s0 <= t) {
                        x = *reinterpret_cast<const float4*>(&Tm[t * NLD + s0]);
                        if (s0 + 1 > t) x.y = 0.f;
                        if (s0 + 2 > t) x.z = 0.f;
                        if (s0 + 3 > t) x.w = 0.f;
                    }
                    return x;
                };
                emit(t_lo, (t_lo < 32 && c4 < 8) ? copy_of(t_lo) : make_float4(0.f, 0.f, 0.f, 0.f));
                const int t = 32 + t_lo, cq2 = c4 & 7;
                float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
                for (int s2 = c4 >> 3; s2 <= t_lo; s2 += 2) {
                    const float tv = Tm[t * NLD + 32 + s2];
                    const float4 yv = *reinterpret_cast<const float4*>(&Y2[s2 * 36 + 4 * cq2]);
                    z.x = fmaf(tv, yv.x, z.x);
                    z.y = fmaf(tv, yv.y, z.y);
                    z.z = fmaf(tv, yv.z, z.z);
                    z.w = fmaf(tv, yv.w, z.w);
                }
                z.x += __shfl_xor_sync(0xffffffffu, z.x, 8);
                z.y += __shfl_xor_sync(0xffffffffu, z.y, 8);
                z.z += __shfl_xor_sync(0xffffffffu, z.z, 8);
                z.w += __shfl_xor_sync(0xffffffffu, z.w, 8);
                emit(t, c4 < 8 ? make_float4(-z.x, -z.y, -z.z, -z.w) : copy_of(t));
            }
        }
        fence_async_smem();  // the image tiles are read by MMA 2 and the bulk store
        fence_before();
        bar_named(kPrepBar, kThreads);
        fence_after();
        // ---- MMA 2: W^T = KG T_b^T (hi*hi + hi*lo + lo*hi)
        if (tid == 0) {
            const uint32_t idk = idesc_bf16(128, 64, false, false, false);
#pragma unroll
            for (int pass = 0; pass < 3; ++pass) {
                const uint32_t a = tmem + (pass == 2 ? PT_KG_LO : PT_KG_HI);
                const uint32_t b = sb4 + (PR_IMG + OP_TB + (pass == 1 ? 8192u : 0u)) / 16;
#pragma unroll
                for (int s = 0; s < 4; ++s)
                    mma_ta(tmem + PT_W, a + 8 * s, desc_k4(b, 64, s), idk, (pass | s) != 0);
            }
            commit(mbar);
        }
        {
            const bool ok2 = mbar_wait(mbar, phase, kWaitLimit);
            phase ^= 1;
            fence_after();
            if (bar_named_or(kPrepBar, kThreads, !ok2)) {
                timed_out = true;
                break;
            }
        }
        // ---- W^T (lanes i, columns t) -> -W operand (B, MN-major [i][t]) hi/lo
        {
            float v[16];
            ld16(tl + PT_W + cq * 16, v);
#pragma unroll
            for (int q = 0; q < 16; ++q) v[q] = -v[q];
#pragma unroll
            for (int c8 = 0; c8 < 2; ++c8) {
                uint4 hi, lo;
                split8p(v + 8 * c8, hi, lo);
                const int t = cq * 16 + 8 * c8;
                st16(sm, PR_IMG + OP_QW + 16384 + chunk_mn(t, row, 1024, 1024), hi);
                st16(sm, PR_IMG + OP_QW + 32768 + chunk_mn(t, row, 1024, 1024), lo);
            }
        }
        fence_async_smem();
        fence_before();
        bar_named(kPrepBar, kThreads);
        fence_after();
        // ---- the block image -> the workspace, by bulk copies the next item does not wait for,
        //      one per issuing thread (lane 0 of warps 7-9), each in its own bulk group
        if (store_lane) {
            if (warp == 7) {
                bulk_store(blk, sb + PR_IMG, opa_bytes(kBf16Out));
            } else if constexpr (kBf16Out) {
                if (warp == 8) bulk_store(blk + OP_KTP, sb + PR_IMG + OP_KTP, OPB1_BYTES_BF16);
                else bulk_store(blk + OP_KTLO, sb + PR_IMG + OP_KTLO, OPB2_BYTES_BF16);
            } else {
                if (warp == 8) bulk_store(blk + OP_KTP, sb + PR_IMG + OP_KTP, OP_BYTES - OP_KTP);
            }
            bulk_commit();
        }
        cur = nxt;
    }
    if (store_lane) bulk_wait_all();  // the image stores have read shared memory and landed
    timed_out = bar_named_or(kPrepBar, kThreads, timed_out);
    if (timed_out) {
        if (tid == 0) report(p.dev_status, KDA_DEV_TIMEOUT);
        mbar_wait(mbar, phase ^ 1u, kWaitLimit);  // the phase that timed out, bounded
        if (qk_pending) mbar_wait(mbar_qk, phase_qk, kWaitLimit);
        mbar_wait(mbar_qk, phase_qk ^ 1u, kWaitLimit);
        if (g_pending) mbar_wait(mbar_g, phase_g, kWaitLimit);
        mbar_wait(mbar_g, phase_g ^ 1u, kWaitLimit);
    }
    fence_before();
    bar_named(kPrepBar, kThreads);
    fence_after();
    if (warp == 0) tmem_dealloc(tmem, PT_COLS);
}

template <bool kBf16Out, bool kF32In>
__global__ void __launch_bounds__(kThreads, 1) prefill_prep_kernel(const __grid_constant__ CUtensorMap qmap,
                                                                   const __grid_constant__ CUtensorMap kmap,
                                                                   const __grid_constant__ CUtensorMap gmap,
                                                                   PrefillArgs p, const int32_t* __restrict__ plan,
                                                                   int64_t n_max, uint8_t* __restrict__ ops,
                                                                   int64_t c_begin, int64_t c_end) {
    prep_body<kBf16Out, kF32In>(&qmap, &kmap, &gmap, p, plan, n_max, ops, blockIdx.x, gridDim.x, c_begin, c_end);
}

// ----------------------------------------------------------------------------
// sweep: one (sequence, head) through its chunks, state in TMEM

constexpr uint32_t SW_OPS = 0;                   // operand block image (parts A and B)
// V, MN-major (two 64-channel boxes, 128-byte swizzled), one buffer: the next chunk's copy is
// issued only after MMA 3, which ends after this chunk's U~ (the one MMA reading V).  fp32
// activations use the second 16 KiB for the lo half of V's bf16 split.
constexpr uint32_t SW_V = SW_OPS + OP_BYTES;
constexpr uint32_t SW_OST = SW_V + 32768;        // bf16 output rows [64][128], two buffers
constexpr uint32_t SW_RED = SW_OST + 32768;      // token path: partial row sums [2][4][128] fp32
constexpr uint32_t SW_MISC = SW_RED + 4096;
constexpr uint32_t SW_SMEM = SW_MISC + 8192 + 1024;
// token path (a flagged chunk): raw q, k (and g for bf16) over the part-A region, alpha over part B
constexpr uint32_t SW_RAW_Q = SW_OPS, SW_RAW_K = SW_OPS + 16384, SW_RAW_G = SW_OPS + 32768;
constexpr uint32_t SW_RAW_Q32 = SW_OPS, SW_RAW_K32 = SW_OPS + 32768;  // fp32 rows [t][128]
constexpr uint32_t SW_ALPHA = SW_OPS + OP_KTP;
static_assert(SW_RAW_G + 16384 <= SW_OPS + OP_GAM, "raw tiles overlap the flag word");
static_assert(SW_RAW_K32 + 32768 <= SW_OPS + OP_GAM, "fp32 raw tiles overlap the flag word");
static_assert(SW_ALPHA + 32768 <= SW_OPS + OP_BYTES, "alpha table overlaps the V buffers");
static_assert(SW_SMEM <= 232448, "sweep shared memory plan exceeds the per-CTA limit");

// TMEM columns (512): as the single-pass kernel
constexpr uint32_t TM_S = 0;                        // S^T, fp32, 128 columns
constexpr uint32_t TM_O = 128;                      // O^T
constexpr uint32_t TM_UA = 192, TM_UB = 256;        // U^T = U_a + U_b (hi and lo T_b parts)
constexpr uint32_t TM_SA_HI = 320, TM_SA_LO = 384;  // S^T [c][i] bf16 hi/lo A operand, K = 128
constexpr uint32_t TM_U_HI = 448, TM_U_LO = 480;    // U^T [c][s] bf16 hi/lo A operand, K = 64
constexpr uint32_t TM_COLS = 512;

constexpr int kIssuerWarp = 16;                  // after the 16 compute warps
constexpr int kSweepThreads = kThreads + 32;

// What a sweep computes over its chunk range.  Across a chunk the state map is affine,
// S' = (Diag(e^{G_63}) - K~^T W) S + K~^T U~, so a range's end state is Phi S_in + B with
// Phi = the range's product of those matrices and B = its end state from S_in = 0:
//   kSweepOut  the outputs, snapshots and end state from the given start state;
//   kSweepPhi  Phi: the state map from S = I with U~ = 0 (V read as zero); no outputs;
//   kSweepB    B: from S = 0; no outputs.
// (Phi is d_k x d_k and fits the d_k x d_v state's storage because d_k = d_v.)
enum SweepMode { kSweepOut = 0, kSweepPhi = 1, kSweepB = 2 };

// Unit `unit` over its chunks [j_begin, j_end) (chunk index within the sequence), or, when
// n_seg > 0, over segment `seg` of n_seg equal parts of its sequence's chunks (the last one to
// the end).  The state enters from `sc_in` (fp32 [unit][v][k]) when given, else from the
// initial slot (kSweepOut), the identity (kSweepPhi) or zero (kSweepB).  A kSweepOut range that
// reaches the sequence's end writes the final slot; otherwise the end state goes to `sc_out`
// ([unit][v][k]) when given.
template <bool kBf16Out, bool kF32In>
__device__ __forceinline__ void sweep_body(const CUtensorMap* vmap, const CUtensorMap* omap, const PrefillArgs& p,
                                           const int32_t* __restrict__ plan, int64_t n_max,
                                           const uint8_t* __restrict__ ops, int unit, int j_begin, int j_end,
                                           const float* __restrict__ sc_in, float* __restrict__ sc_out,
                                           int mode, int seg = 0, int n_seg = 0) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(sm);
    const uint32_t sb4 = sb >> 4;
    float* s_beta = reinterpret_cast<float*>(sm + SW_MISC);            // 64 (token path)
    float* s_nk = s_beta + 64;                                         // 64: key-row L2 factors (token path)
    float* s_nq = s_nk + 64;                                           // 64: query-row factors x scale
    int* s_trk = reinterpret_cast<int*>(s_nq + 64);                    // kTrack2p
    // MMA, S update, part A + V, part B (one arrival each); S operand and U operand written
    // (one arrival per thread)
    uint64_t* s_mbar = reinterpret_cast<uint64_t*>(s_trk + kTrack2p);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(s_mbar + 6);

    // Roles.  Warps 0-15 (compute) run the TMEM passes: warp w reads lane quarter w % 4 and
    // column quarter w / 4 of a tile.  Warp 16 (issuer) issues every MMA, operand copy, L2
    // prefetch and output store: a single issuing thread that also took part in the passes
    // would put all of that on the serial path of every chunk.
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool issuer = warp == kIssuerWarp;
    const bool lead = issuer && lane == 0;
    const int quarter = warp & 3;
    const int cq = warp >> 2;
    const int row = quarter * 32 + lane;
    const int ci = tid & 127, tq = tid >> 7;
    const int H = p.H;
    const int n = plan[PL_ORDER / 4 + unit / H];
    const int h = unit - (unit / H) * H;

    const int t0 = p.cu_seqlens[n], t1 = p.cu_seqlens[n + 1];
    if (t0 < 0 || t1 < t0 || t1 > p.T_tot || (n == 0 && t0 != 0)) {
        if (tid == 0 && h == 0) report(p.dev_status, KDA_DEV_BAD_SEQLEN);
        return;
    }
    const int L = t1 - t0;
    const int n_chunks = (L + kChunk - 1) / kChunk;
    const int64_t cbase = plan[PL_BASE / 4 + n];
    if (cbase + n_chunks > n_max) {  // sequences overlap in cu_seqlens: no room in the plan
        if (tid == 0 && h == 0) report(p.dev_status, KDA_DEV_BAD_SEQLEN);
        return;
    }
    const int init = p.init_slot ? p.init_slot[n] : -1;
    const int fin = p.final_slot ? p.final_slot[n] : -1;
    if (init >= p.P || fin >= p.P) {
        if (tid == 0 && h == 0) report(p.dev_status, KDA_DEV_BAD_SLOT);
        return;
    }
    // this call's chunks; a range that starts past the sequence's end, or a later segment of an
    // empty sequence, has nothing left to do (the call that reached the end wrote the final state)
    int jb = j_begin, j_last = j_end;
    if (n_seg > 0) {  // n_chunks < 2^25 and seg < 16: the products fit in 32 bits
        jb = n_chunks * seg / n_seg;
        j_last = seg + 1 == n_seg ? INT_MAX : n_chunks * (seg + 1) / n_seg;
    }
    const int je = min(n_chunks, j_last);
    if ((jb > 0 || seg > 0) && jb >= n_chunks) return;
    const bool outputs = mode == kSweepOut;  // outputs and snapshots
    const bool zero_v = mode == kSweepPhi;   // U~ = T_b V with V read as zero
    const bool to_pool = outputs && j_last >= n_chunks;
    const bool to_sc = !to_pool && sc_out != nullptr;
    for (int m = tid; m < p.M; m += kSweepThreads) {
        const int jj = p.track[(size_t)n * p.M + m];
        const bool ok = jj >= -1 && jj < n_chunks;
        if (!ok && h == 0) report(p.dev_status, KDA_DEV_BAD_TRACK);
        s_trk[m] = ok ? jj : -1;
    }

    if (warp == 0) tmem_alloc(smem_u32(s_tmem), TM_COLS);
    if (lead) {
        for (int b = 0; b < 4; ++b) mbar_init(smem_u32(s_mbar + b), 1);
        mbar_init(smem_u32(s_mbar + 4), kThreads);  // one arrival per compute thread
        mbar_init(smem_u32(s_mbar + 5), kThreads);
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t mbar = smem_u32(s_mbar), mbar_s = smem_u32(s_mbar + 1);
    const uint32_t mbar_a = smem_u32(s_mbar + 2), mbar_b = smem_u32(s_mbar + 3);
    const uint32_t mbar_s1 = smem_u32(s_mbar + 4), mbar_u = smem_u32(s_mbar + 5);
    uint32_t ph_s1 = 0, ph_u = 0;
    // the next chunk with a snapshot request
    int next_snap = outputs ? next_tracked(s_trk, p.M, jb - 1) : 0x7fffffff;
    // every thread tracks the phases in step; the waits are done by the threads that need them
    uint32_t phase = 0, phase_s = 0, phase_a = 0, phase_b = 0;
    bool pending_s = false;               // state update issued, not yet waited on
    bool pend_a = false, pend_b = false;  // copies issued, not yet waited on
    const uint32_t na = opa_bytes(kBf16Out), nb = opb_bytes(kBf16Out);
    auto block_of = [&](int jj) { return ops + ((size_t)(cbase + jj) * H + h) * OP_BYTES; };
    // part A of chunk jj and, for bf16 activations, its V tile (two 64-channel boxes of the
    // tensor map over v, 128-byte swizzled: the MN-major MMA operand), one barrier.  fp32 V is
    // split into bf16 hi/lo tiles by the compute threads at the chunk's start instead.
    auto load_a = [&](int jj) {
        const bool tma_v = !kF32In && !zero_v;
        mbar_expect_tx(mbar_a, na + (tma_v ? 16384u : 0u));
        bulk_load(sb + SW_OPS, block_of(jj), na, mbar_a);
        if (tma_v) {
            tma_load_2d(sb + SW_V, vmap, h * kD, t0 + jj * kChunk, mbar_a);
            tma_load_2d(sb + SW_V + 8192, vmap, h * kD + 64, t0 + jj * kChunk, mbar_a);
        }
    };
    // part B of chunk jj: one bulk copy, or two around the unused P lo tile
    auto load_b = [&](int jj) {
        mbar_expect_tx(mbar_b, nb);
        if constexpr (kBf16Out) {
            bulk_load(sb + SW_OPS + OP_KTP, block_of(jj) + OP_KTP, OPB1_BYTES_BF16, mbar_b);
            bulk_load(sb + SW_OPS + OP_KTLO, block_of(jj) + OP_KTLO, OPB2_BYTES_BF16, mbar_b);
        } else {
            bulk_load(sb + SW_OPS + OP_KTP, block_of(jj) + OP_KTP, nb, mbar_b);
        }
    };
    // chunk jj's operand block and V into L2, so that its shared-memory copies (issued when the
    // single buffers free up) wait on L2 rather than on HBM
    auto prefetch_l2 = [&](int jj) {
        const uint8_t* b2 = block_of(jj);
        bulk_prefetch_l2(b2, opa_bytes(kBf16Out));
        bulk_prefetch_l2(b2 + OP_KTP, OP_BYTES - OP_KTP);
        if (!kF32In && !zero_v) {
            tma_prefetch_2d(vmap, h * kD, t0 + jj * kChunk);
            tma_prefetch_2d(vmap, h * kD + 64, t0 + jj * kChunk);
        }
    };
    // U~^T = V^T [T_b hi; T_b lo]^T into [U_a | U_b]; fp32 V adds V_lo^T T_b hi^T into U_a
    auto issue_u_tilde = [&]() {
        const uint32_t idv = idesc_bf16(128, 128, true, false, false);
#pragma unroll
        for (int s = 0; s < 4; ++s)
            mma(tmem + TM_UA, desc_mn4(sb4 + SW_V / 16, 8192, 1024, s),
                desc_k4(sb4 + (SW_OPS + OP_TB) / 16, 128, s), idv, s != 0);
        if constexpr (kF32In) {
            const uint32_t idv1 = idesc_bf16(128, 64, true, false, false);
#pragma unroll
            for (int s = 0; s < 4; ++s)
                mma(tmem + TM_UA, desc_mn4(sb4 + (SW_V + 16384) / 16, 8192, 1024, s),
                    desc_k4(sb4 + (SW_OPS + OP_TB) / 16, 128, s), idv1, 1u);
        }
    };

    // ---- initial state into TMEM; O columns cleared (MMA 3 accumulates into them)
    if (!issuer) {
        const size_t S0 = init >= 0 ? state_elem(init, H, h) + (size_t)row * kD : 0;
        const int col0 = cq * 32;
        float v[32];
#pragma unroll
        for (int jj = 0; jj < 32; jj += 4) {
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (sc_in != nullptr)
                x = *reinterpret_cast<const float4*>(sc_in + ((size_t)unit * kD + row) * kD + col0 + jj);
            else if (outputs && init >= 0)
                x = state_load4(p.pool, S0 + col0 + jj, p.st);
            v[jj] = x.x;
            v[jj + 1] = x.y;
            v[jj + 2] = x.z;
            v[jj + 3] = x.w;
        }
        if (sc_in == nullptr && mode == kSweepPhi) {
#pragma unroll
            for (int q = 0; q < 32; ++q) v[q] = col0 + q == row ? 1.f : 0.f;
        }
        st32(tl + TM_S + col0, v);
        if (zero_v && !kF32In) {
            // V stays zero: no copy ever lands in its buffer (a partial chunk's clearing writes
            // zeros as well)
            for (int e = tid; e < 2048; e += kThreads) st16(sm, SW_V + e * 16, make_uint4(0, 0, 0, 0));
            fence_async_smem();
        }
        float z[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) z[q] = 0.f;
        st16f(tl + TM_O + cq * 16, z);
        wait_st();
    }
    if (je > jb) {
        if (lead) {
            load_a(jb);
            load_b(jb);
            if (jb + 1 < je) prefetch_l2(jb + 1);
        }
        pend_a = pend_b = true;
    }
    fence_before();
    __syncthreads();
    fence_after();

    bool timed_out = false;
    // bf16 output rows staged in shared memory; the issuer warp stores them after the next barrier
    bool o_pending = false;
    int o_c0 = 0, o_Lc = 0;
    uint32_t o_buf = 0;
    auto store_o_rows = [&]() {  // issuer warp: a full chunk as one tensor store, else per row
        if (!o_pending) return;
        bulk_wait_read_all();  // the stores of two chunks ago have read that staging buffer
        if (o_Lc == kChunk) {
            if (lane == 0) tma_store_2d(omap, h * kD, o_c0, sb + SW_OST + o_buf * 16384);
        } else {
            for (int t = lane; t < o_Lc; t += 32)
                bulk_store(static_cast<__nv_bfloat16*>(p.out) + ((size_t)(o_c0 + t) * H + h) * kD,
                           sb + SW_OST + o_buf * 16384 + t * 256, 256);
        }
        bulk_commit();
        o_pending = false;
    };

    // every exit from the loop is decided at a barrier (uniform across the CTA)
    for (int j = jb; j < je; ++j) {
        const int c0 = t0 + j * kChunk;
        const int Lc = min(kChunk, t1 - c0);
        const bool more = j + 1 < je;
        const bool snap_here = j == next_snap;
        // the previous chunk's state update: the compute warps read S next; its end frees part B
        if (pending_s) {
            if (!mbar_wait(mbar_s, phase_s, kWaitLimit)) timed_out = true;
            phase_s ^= 1;
            pending_s = false;
        }
        if (!timed_out && j > jb) {
            if (lead) load_b(j);
            pend_b = true;
        }
        fence_after();
        // ---- state pass, first half: S_j -> bf16 hi/lo A operand in TMEM (16 of this thread's 32
        //      columns at a time), while part A may still be landing; a chunk that turns out to
        //      take the token path reads S itself and leaves the operand unused
        if (!timed_out && !issuer) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                float v[16];
                ld16(tl + TM_S + cq * 32 + 16 * hh, v);
                uint32_t sh[8], sl[8];
#pragma unroll
                for (int q2 = 0; q2 < 8; ++q2) split2p(v[2 * q2], v[2 * q2 + 1], sh[q2], sl[q2]);
                st8u(tl + TM_SA_HI + cq * 16 + 8 * hh, sh);
                st8u(tl + TM_SA_LO + cq * 16 + 8 * hh, sl);
            }
            wait_st();
        }
        if (!timed_out) {
            if (!mbar_wait(mbar_a, phase_a, kWaitLimit)) timed_out = true;
            phase_a ^= 1;
            pend_a = false;
        }
        const bool partial = Lc < kChunk;
        // V written by the compute threads (fp32 split, or rows past a partial chunk cleared):
        // U~ then waits for their arrivals on mbar_s1
        const bool v_by_threads = kF32In || partial;
        // the token path's first barrier decides a timeout for every thread; the chunk path
        // decides at its barrier after MMA 3
        const bool flagged = !timed_out && *reinterpret_cast<const int32_t*>(sm + SW_OPS + OP_FLAG) != 0;

        if (!flagged) {
            if constexpr (kF32In) {
                if (!timed_out && !issuer) {
                    // fp32 V -> bf16 hi/lo tiles in the TMA box layout (rows past the sequence 0)
                    const float* gv = static_cast<const float*>(p.v);
#pragma unroll
                    for (int e = tid; e < 64 * 16; e += kThreads) {
                        const int t = e >> 4, g8 = e & 15;
                        float x[8];
                        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
                        if (t < Lc && !zero_v) {
                            const float4* src = reinterpret_cast<const float4*>(gv + ((size_t)(c0 + t) * H + h) * kD + 8 * g8);
                            a = __ldg(src);
                            b = __ldg(src + 1);
                        }
                        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
                        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
                        uint4 hi, lo;
                        split8p(x, hi, lo);
                        const uint32_t off = chunk_mn(8 * g8, t, 8192, 1024);
                        st16(sm, SW_V + off, hi);
                        st16(sm, SW_V + 16384 + off, lo);
                    }
                    fence_async_smem();
                }
            } else if (partial && !timed_out && !issuer) {
                // V rows past the sequence (the next sequence's, or zero-filled past T_tot) -> 0,
                // so that no other row's values (possibly non-finite) enter this chunk
                for (int e = tid; e < 2 * 64 * 8; e += kThreads) {
                    const int a = e >> 9, t = (e >> 3) & 63, c16 = e & 7;
                    if (t >= Lc)
                        st16(sm, SW_V + a * 8192 + (t >> 3) * 1024 + (t & 7) * 128 + c16 * 16,
                             make_uint4(0, 0, 0, 0));
                }
                fence_async_smem();
            }
            if (!issuer) {
                // the S operand (and V, where the threads wrote it) is ready for MMA 3
                fence_before();
                mbar_arrive(mbar_s1);
            }
            // ---- MMA 3 (lead, once every compute thread's S operand is in TMEM): [O | U_a | U_b]
            //      += S_hi^T [QG; -W_hi; -W_lo]^T, [O | U_a] += S_lo^T [QG; -W_hi]^T; fp32 outputs
            //      also S_hi^T QG_lo^T.  U^T = U_a + U_b.  U~ runs first (it needs only this
            //      chunk's operands), then the L2 prefetch of the next chunk.
            if (lead) {
                if (!v_by_threads) issue_u_tilde();
                if (mbar_wait(mbar_s1, ph_s1, kWaitLimit)) {
                    fence_after();
                    if (v_by_threads) issue_u_tilde();
                    const uint32_t id3 = idesc_bf16(128, 192, false, true, false);
                    const uint32_t id2 = idesc_bf16(128, 128, false, true, false);
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        mma_ta(tmem + TM_O, tmem + TM_SA_HI + 8 * s,
                               desc_mn4(sb4 + (SW_OPS + OP_QW) / 16, 16384, 1024, s), id3, 1u);
#pragma unroll
                    for (int s = 0; s < 8; ++s)
                        mma_ta(tmem + TM_O, tmem + TM_SA_LO + 8 * s,
                               desc_mn4(sb4 + (SW_OPS + OP_QW) / 16, 16384, 1024, s), id2, 1u);
                    if constexpr (!kBf16Out) {
                        const uint32_t id1 = idesc_bf16(128, 64, false, true, false);
#pragma unroll
                        for (int s = 0; s < 8; ++s)
                            mma_ta(tmem + TM_O, tmem + TM_SA_HI + 8 * s,
                                   desc_mn4(sb4 + (SW_OPS + OP_QGLO) / 16, 16384, 1024, s), id1, 1u);
                    }
                    commit(mbar);
                } else {
                    timed_out = true;  // the others' MMA 3 wait below then gives up as well
                }
                // the next chunk into L2, under MMA 3 (the start prefetched chunk jb + 1): one
                // chunk ahead measured level with two on the batched call and ~1 % faster on
                // long sequences; three ahead was 11 % slower, none 3 %
                if (j > jb && j + 1 < je) prefetch_l2(j + 1);
            }
            ph_s1 ^= 1;
            // ---- state pass, second half (under MMA 3, which does not touch the S columns):
            //      the snapshot of S_j, then S <- S Diag(e^{G_63})
            if (!issuer) {
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    const int col0 = cq * 32 + 16 * hh;
                    float v[16];
                    ld16(tl + TM_S + col0, v);
                    if (snap_here) {
                        for (int m = 0; m < p.M; ++m) {
                            if (s_trk[m] != j) continue;
                            const size_t snap = state_elem((int64_t)n * p.M + m, H, h) + (size_t)row * kD + col0;
#pragma unroll
                            for (int q4 = 0; q4 < 16; q4 += 4)
                                state_store4(p.track_state, snap + q4,
                                             make_float4(v[q4], v[q4 + 1], v[q4 + 2], v[q4 + 3]), p.st);
                        }
                    }
                    const float2* gm2 = reinterpret_cast<const float2*>(sm + SW_OPS + OP_GAM + col0 * 4);
#pragma unroll
                    for (int q2 = 0; q2 < 8; ++q2) {
                        const float2 x = __fmul2_rn(make_float2(v[2 * q2], v[2 * q2 + 1]), gm2[q2]);
                        v[2 * q2] = x.x;
                        v[2 * q2 + 1] = x.y;
                    }
                    st16f(tl + TM_S + col0, v);
                }
                wait_st();
            }
            fence_async_smem();  // part A's reads are done before the next chunk's copy into it
            if (issuer) bulk_wait_read_all();  // row stores of two chunks ago: that staging is free
            const bool ok3 = mbar_wait(mbar, phase, kWaitLimit);
            phase ^= 1;
            fence_before();
            // the chunk's one CTA barrier: MMA 3 has ended for everyone and every thread is past
            // its reads of part A and its writes of the previous chunk's output rows
            if (__syncthreads_or(!ok3 || timed_out)) {
                timed_out = true;
                break;
            }
            fence_after();
            // part A is free from here (MMA 3 ended and every reader is past the barrier); the next
            // chunk's part A and V are requested once MMA 4 is issued (measured ~2 % faster on one
            // long sequence than requesting them here).  The previous chunk's staged output rows
            // leave now.
            if (issuer) store_o_rows();
            // ---- U^T (lanes c, columns s) -> bf16 hi/lo A operand in TMEM; arrive on mbar_u
            if (!issuer) {
                uint32_t ra[16], rb[16];
                ld16_issue(tl + TM_UA + cq * 16, ra);
                ld16_issue(tl + TM_UB + cq * 16, rb);
                wait_ld();
                float v[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) v[q] = __uint_as_float(ra[q]) + __uint_as_float(rb[q]);
                uint32_t uh[8], ul[8];
#pragma unroll
                for (int q2 = 0; q2 < 8; ++q2) split2p(v[2 * q2], v[2 * q2 + 1], uh[q2], ul[q2]);
                st8u(tl + TM_U_HI + cq * 8, uh);
                st8u(tl + TM_U_LO + cq * 8, ul);
                wait_st();
                fence_before();
                mbar_arrive(mbar_u);
            }
            if (more) pend_a = true;
            // ---- MMA 4 (lead, once every thread's U operand is in TMEM and part B has landed):
            //      [S | O] += U_hi^T [KT_hi; P]^T (N = 192); then the rest of the state update,
            //      S^T += U_lo^T KT_hi + U_hi^T KT_lo
            if (lead) {
                if (mbar_wait(mbar_u, ph_u, kWaitLimit) && mbar_wait(mbar_b, phase_b, kWaitLimit)) {
                    fence_after();
                    const uint32_t id3 = idesc_bf16(128, 192, false, false, false);
                    const uint32_t id2 = idesc_bf16(128, 128, false, false, false);
                    const uint32_t ktp = sb4 + (SW_OPS + OP_KTP) / 16;
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        mma_ta(tmem + TM_S, tmem + TM_U_HI + 8 * s, desc_k4(ktp, 192, s), id3, 1u);
                    if constexpr (!kBf16Out) {
                        const uint32_t id1 = idesc_bf16(128, 64, false, false, false);
#pragma unroll
                        for (int s = 0; s < 4; ++s)
                            mma_ta(tmem + TM_S, tmem + TM_U_LO + 8 * s, desc_k4(ktp, 192, s), id3, 1u);
#pragma unroll
                        for (int s = 0; s < 4; ++s)
                            mma_ta(tmem + TM_O, tmem + TM_U_HI + 8 * s,
                                   desc_k4(sb4 + (SW_OPS + OP_PLO) / 16, 64, s), id1, 1u);
                    }
                    commit(mbar);  // the outputs
                    if constexpr (kBf16Out) {
#pragma unroll
                        for (int s = 0; s < 4; ++s)
                            mma_ta(tmem + TM_S, tmem + TM_U_LO + 8 * s, desc_k4(ktp, 128, s), id2, 1u);
                    }
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        mma_ta(tmem + TM_S, tmem + TM_U_HI + 8 * s,
                               desc_k4(sb4 + (SW_OPS + OP_KTLO) / 16, 128, s), id2, 1u);
                    commit(mbar_s);
                    if (more) load_a(j + 1);  // lands under MMA 4 and the output pass
                } else {
                    timed_out = true;  // the others' output wait below then gives up as well
                }
            }
            ph_u ^= 1;
            phase_b ^= 1;
            pend_b = false;
            pending_s = true;
            const bool ok4 = mbar_wait(mbar, phase, kWaitLimit);
            phase ^= 1;
            fence_after();
            if (!ok4) timed_out = true;  // decided at the next chunk's barrier
            // ---- O^T (lanes c, columns t) -> out[t][h][c]: bf16 rows staged for warp 1's
            //      stores after the next chunk's barrier, fp32 straight from registers (a warp
            //      stores 32 consecutive value channels per t).  The O columns are cleared for
            //      the next MMA 3 (ordered before it by the next chunk's arrival on mbar_s1).
            if (ok4 && !issuer && outputs) {
                float v[16];
                ld16(tl + TM_O + cq * 16, v);
                if constexpr (kBf16Out) {
                    __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(sm + SW_OST + (uint32_t)(j & 1) * 16384);
#pragma unroll
                    for (int q = 0; q < 16; ++q) ob[(cq * 16 + q) * kD + row] = __float2bfloat16_rn(v[q]);
                    fence_async_smem();
                } else {
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int t = cq * 16 + q;
                        if (t < Lc) store1<false>(p.out, ((size_t)(c0 + t) * H + h) * kD + row, v[q]);
                    }
                }
#pragma unroll
                for (int q = 0; q < 16; ++q) v[q] = 0.f;
                st16f(tl + TM_O + cq * 16, v);
                wait_st();
            } else if (ok4 && !issuer) {
                // no outputs: the O columns are only cleared for the next MMA 3
                float z[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) z[q] = 0.f;
                st16f(tl + TM_O + cq * 16, z);
                wait_st();
            }
            if (kBf16Out && outputs) {
                o_pending = true;
                o_c0 = c0;
                o_Lc = Lc;
                o_buf = (uint32_t)(j & 1);
            }
        } else {
            // ---- token path: this chunk on CUDA cores, exactly in fp32.  Part B's region takes
            //      the alpha table, part A's the raw tiles: wait for part B's copy to land first.
            const bool okb = mbar_wait(mbar_b, phase_b, kWaitLimit);
            phase_b ^= 1;
            pend_b = false;
            if (__syncthreads_or(!okb)) {
                timed_out = true;
                break;
            }
            if (issuer) store_o_rows();  // the previous chunk's rows, if staged
            {
                if constexpr (kF32In) {
                    const float* gq = static_cast<const float*>(p.q);
                    const float* gk = static_cast<const float*>(p.k);
                    for (int it = tid; it < 64 * 32; it += kSweepThreads) {
                        const int t = it >> 5, ch = it & 31;
                        const bool ok = t < Lc;
                        const size_t e = ok ? ((size_t)(c0 + t) * H + h) * kD + ch * 4 : 0;
                        const uint32_t nbt = ok ? 16u : 0u;
                        cp_async16(sb + SW_RAW_Q32 + t * 512 + ch * 16, gq + e, nbt);
                        cp_async16(sb + SW_RAW_K32 + t * 512 + ch * 16, gk + e, nbt);
                    }
                } else {
                    const __nv_bfloat16* gq = static_cast<const __nv_bfloat16*>(p.q);
                    const __nv_bfloat16* gk = static_cast<const __nv_bfloat16*>(p.k);
                    const __nv_bfloat16* gg = static_cast<const __nv_bfloat16*>(p.gate_raw);
                    for (int it = tid; it < 64 * 16; it += kSweepThreads) {
                        const int t = it >> 4, ch = it & 15;
                        const bool ok = t < Lc;
                        const size_t e = ok ? ((size_t)(c0 + t) * H + h) * kD + ch * 8 : 0;
                        const uint32_t nbt = ok ? 16u : 0u;
                        cp_async16(sb + SW_RAW_Q + t * 256 + ch * 16, gq + e, nbt);
                        cp_async16(sb + SW_RAW_K + t * 256 + ch * 16, gk + e, nbt);
                        cp_async16(sb + SW_RAW_G + t * 256 + ch * 16, gg + e, nbt);
                    }
                }
                cp_async_commit();
                if (tid < 64) {
                    const size_t bi = (size_t)(c0 + min(tid, Lc - 1)) * H + h;
                    const float braw = kF32In ? __ldg(static_cast<const float*>(p.beta_raw) + bi)
                                              : __uint_as_float((uint32_t)__ldg(static_cast<const unsigned short*>(p.beta_raw) + bi) << 16);
                    s_beta[tid] = tid < Lc ? beta_act(braw, p.flags) : 0.f;
                }
                cp_async_wait_all();
                __syncthreads();
            }
            // raw key / query element (t, i) of this chunk, and the raw value (t, c)
            auto raw_k = [&](int t, int i) {
                if constexpr (kF32In) return *reinterpret_cast<const float*>(sm + SW_RAW_K32 + t * 512 + i * 4);
                else return bf16_at(sm, SW_RAW_K + t * 256 + i * 2);
            };
            auto raw_q = [&](int t, int i) {
                if constexpr (kF32In) return *reinterpret_cast<const float*>(sm + SW_RAW_Q32 + t * 512 + i * 4);
                else return bf16_at(sm, SW_RAW_Q + t * 256 + i * 2);
            };
            if (!issuer) {
                // the factors the key / query rows are used with (1 and scale without the flag)
                const bool l2 = (p.flags & KDA_QK_L2NORM) != 0;
#pragma unroll
                for (int tt = 0; tt < 4; ++tt) {
                    const int t = 4 * warp + tt;
                    float fk = 1.f, fq = p.scale;
                    if (l2) {
                        float4 kx, qx;
                        if constexpr (kF32In) {
                            kx = *reinterpret_cast<const float4*>(sm + SW_RAW_K32 + t * 512 + lane * 16);
                            qx = *reinterpret_cast<const float4*>(sm + SW_RAW_Q32 + t * 512 + lane * 16);
                        } else {
                            kx = State<kStateBF16>::widen(*reinterpret_cast<const uint2*>(sm + SW_RAW_K + t * 256 + lane * 8));
                            qx = State<kStateBF16>::widen(*reinterpret_cast<const uint2*>(sm + SW_RAW_Q + t * 256 + lane * 8));
                        }
                        float sk = f4_dot(kx, kx), sq = f4_dot(qx, qx);
                        warp_sum2(sk, sq);
                        fk = l2norm_factor(sk);
                        fq = l2norm_factor(sq) * p.scale;
                    }
                    if (lane == 0) {
                        s_nk[t] = fk;
                        s_nq[t] = fq;
                    }
                }
            }
            float* alpha = reinterpret_cast<float*>(sm + SW_ALPHA);
            if (!issuer) {
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int t = 16 * tq + u;
                    float graw = 0.f;
                    if constexpr (kF32In) {
                        if (t < Lc) graw = __ldg(static_cast<const float*>(p.gate_raw) + ((size_t)(c0 + t) * H + h) * kD + ci);
                    } else {
                        graw = bf16_at(sm, SW_RAW_G + t * 256 + ci * 2);
                    }
                    alpha[t * kD + ci] = t < Lc ? alpha_of(graw, p.flags) : 1.f;
                }
            }
            fence_before();
            __syncthreads();
            fence_after();
            {
                // thread (row c, column quarter) keeps 32 state columns in registers; the four
                // partial row dot products meet in shared memory
                float* red = reinterpret_cast<float*>(sm + SW_RED);  // [2 dots][4 quarters][128]
                const int c = row;
                float sv[32];
                if (!issuer) {
                    ld32(tl + TM_S + cq * 32, sv);
                    for (int m = 0; m < (snap_here ? p.M : 0); ++m) {
                        if (s_trk[m] != j) continue;
                        const size_t snap = state_elem((int64_t)n * p.M + m, H, h) + (size_t)c * kD + cq * 32;
#pragma unroll
                        for (int q4 = 0; q4 < 32; q4 += 4)
                            state_store4(p.track_state, snap + q4,
                                         make_float4(sv[q4], sv[q4 + 1], sv[q4 + 2], sv[q4 + 3]), p.st);
                    }
                }
                for (int t = 0; t < Lc; ++t) {
                    float d1 = 0.f;
                    if (!issuer) {
                        const float fk = s_nk[t];
#pragma unroll
                        for (int q = 0; q < 32; ++q) {
                            const int i = cq * 32 + q;
                            sv[q] *= alpha[t * kD + i];
                            d1 = fmaf(sv[q], raw_k(t, i) * fk, d1);
                        }
                        red[cq * 128 + c] = d1;
                    }
                    __syncthreads();
                    if (!issuer) {
                        d1 = (red[c] + red[128 + c]) + (red[256 + c] + red[384 + c]);
                        float vt = 0.f;
                        if (!zero_v) {
                            if constexpr (kF32In)
                                vt = __ldg(static_cast<const float*>(p.v) + ((size_t)(c0 + t) * H + h) * kD + c);
                            else
                                vt = bf16_at(sm, SW_V + chunk_mn(c & ~7, t, 8192, 1024) + (c & 7) * 2);
                        }
                        const float uu = s_beta[t] * (vt - d1);
                        float o = 0.f;
                        const float fk = s_nk[t], fq = s_nq[t];
#pragma unroll
                        for (int q = 0; q < 32; ++q) {
                            const int i = cq * 32 + q;
                            sv[q] = fmaf(uu, raw_k(t, i) * fk, sv[q]);
                            o = fmaf(sv[q], raw_q(t, i) * fq, o);
                        }
                        red[512 + cq * 128 + c] = o;
                    }
                    __syncthreads();
                    if (!issuer && cq == 0 && outputs)
                        store1<kBf16Out>(p.out, ((size_t)(c0 + t) * H + h) * kD + c,
                                         (red[512 + c] + red[640 + c]) + (red[768 + c] + red[896 + c]));
                    __syncthreads();  // red is rewritten by the next token
                }
                if (!issuer) {
                    st32(tl + TM_S + cq * 32, sv);
                    wait_st();
                }
            }
            // the regions were written by the generic proxy; the next copies overwrite them
            fence_async_smem();
            fence_before();
            __syncthreads();
            fence_after();
            if (lead && more) load_a(j + 1);
            if (more) pend_a = true;
        }
        if (snap_here) next_snap = next_tracked(s_trk, p.M, j);
    }

    if (pending_s && !timed_out) {
        if (!mbar_wait(mbar_s, phase_s, kWaitLimit)) timed_out = true;
        pending_s = false;
    }
    fence_before();
    timed_out = __syncthreads_or(timed_out);
    fence_after();
    if (issuer) {
        if (!timed_out) store_o_rows();  // the last chunk's rows
        bulk_wait_all();                 // every row store has read its stage and landed
    }
    if (timed_out) {
        if (tid == 0) report(p.dev_status, KDA_DEV_TIMEOUT);
        // give in-flight MMAs and copies a bounded chance to drain before TMEM and shared memory
        // are released: the last phase waited on of each barrier (a wait on a completed phase
        // returns at once) and anything issued but not yet waited on
        mbar_wait(mbar, phase ^ 1u, kWaitLimit);
        mbar_wait(mbar_s, phase_s ^ 1u, kWaitLimit);
        if (pending_s) mbar_wait(mbar_s, phase_s, kWaitLimit);
        if (pend_a) mbar_wait(mbar_a, phase_a, kWaitLimit);
        if (pend_b) mbar_wait(mbar_b, phase_b, kWaitLimit);
    } else if (to_sc && !issuer) {
        float* sc = sc_out + ((size_t)unit * kD + row) * kD + cq * 32;
        float v[32];
        ld32(tl + TM_S + cq * 32, v);
#pragma unroll
        for (int q4 = 0; q4 < 32; q4 += 4)
            *reinterpret_cast<float4*>(sc + q4) = make_float4(v[q4], v[q4 + 1], v[q4 + 2], v[q4 + 3]);
    } else if (to_pool && fin >= 0 && !issuer) {
        const size_t SD = state_elem(fin, H, h) + (size_t)row * kD;
        const int col0 = cq * 32;
        float v[32];
        ld32(tl + TM_S + col0, v);
#pragma unroll
        for (int q4 = 0; q4 < 32; q4 += 4)
            state_store4(p.pool, SD + col0 + q4, make_float4(v[q4], v[q4 + 1], v[q4 + 2], v[q4 + 3]), p.st);
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 0) tmem_dealloc(tmem, TM_COLS);
}

template <bool kBf16Out, bool kF32In>
__global__ void __launch_bounds__(kSweepThreads, 1) prefill_sweep_kernel(const __grid_constant__ CUtensorMap vmap,
                                                                         const __grid_constant__ CUtensorMap omap,
                                                                         PrefillArgs p, const int32_t* __restrict__ plan,
                                                                         int64_t n_max,
                                                                         const uint8_t* __restrict__ ops, int j_begin,
                                                                         int j_end, const float* __restrict__ sc_in,
                                                                         float* __restrict__ sc_out) {
    sweep_body<kBf16Out, kF32In>(&vmap, &omap, p, plan, n_max, ops, blockIdx.x, j_begin, j_end, sc_in, sc_out,
                                 kSweepOut);
}

// One long sequence: the sweep over chunks [sj_begin, sj_end) on CTAs 0 .. units-1 (one per
// unit) and, on the other CTAs, the prep of the chunks after them, [pc_begin, pc_end).  The two
// halves share no data and never wait on each other; the next launch sweeps what this one
// prepared.
template <bool kBf16Out, bool kF32In>
__global__ void __launch_bounds__(kSweepThreads, 1) prefill_pipe_kernel(
    const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap omap,
    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
    const __grid_constant__ CUtensorMap gmap, PrefillArgs p, const int32_t* __restrict__ plan, int64_t n_max,
    uint8_t* __restrict__ ops, float* __restrict__ scratch, int units, int sj_begin, int sj_end, int64_t pc_begin,
    int64_t pc_end) {
    if ((int)blockIdx.x < units) {
        sweep_body<kBf16Out, kF32In>(&vmap, &omap, p, plan, n_max, ops, blockIdx.x, sj_begin, sj_end,
                                     sj_begin > 0 ? scratch : nullptr, scratch, kSweepOut);
    } else if ((int)threadIdx.x < kThreads) {  // the prep's 512 threads; the 17th warp has no part
        prep_body<kBf16Out, kF32In>(&qmap, &kmap, &gmap, p, plan, n_max, ops, (int)blockIdx.x - units,
                                    (int)gridDim.x - units, pc_begin, pc_end);
    }
}

// ---- long sequences with few heads, chunk segments swept in parallel (a scan over the affine
//      state map)
//
// Each sequence's chunks are cut into P equal segments (the last to the end).  Launch 1 sweeps
// segment 0 from the initial state (outputs included; its end state is segment 1's start) and,
// for every middle segment s = 1 .. P-2, its Phi_s and B_s (two CTAs per (sequence, head)).  The
// combine chains the start states, S_{s+1} = Phi_s S_s + B_s.  Launch 2 sweeps segments
// 1 .. P-1 from those starts, outputs included.  Each chunk of a middle segment is swept three
// times, but P segments run at once.  A unit's segment bounds follow its own sequence's length,
// so sequences of different lengths (or empty ones) share the launches.
constexpr int kMaxSeg = 16;
constexpr int64_t kScanMinChunks = 256;  // per sequence, on average
constexpr int kScanMaxN = 8;

// scratch slot of one kind (0: segment start states, 1: Phi, 2: B) and segment, [unit][v][k]
__host__ __device__ inline float* scan_slot(float* scan, int kind, int seg, int units) {
    return scan + (size_t)(kind * kMaxSeg + seg) * (size_t)units * kD * kD;
}

template <bool kBf16Out, bool kF32In>
__global__ void __launch_bounds__(kSweepThreads, 1) prefill_scan_kernel(
    const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap omap, PrefillArgs p,
    const int32_t* __restrict__ plan, int64_t n_max, const uint8_t* __restrict__ ops, int P,
    float* __restrict__ scan, int units, int second) {
    const int bx = blockIdx.x;
    int unit, seg, mode;
    const float* sc_in = nullptr;
    float* sc_out = nullptr;
    if (!second) {
        if (bx < units) {  // segment 0 from the initial state; its end state starts segment 1
            unit = bx;
            seg = 0;
            sc_out = scan_slot(scan, 0, 1, units);
            mode = kSweepOut;
        } else {  // Phi and B of the middle segments
            const int r = (bx - units) / units, kind = (r & 1) ? 2 : 1;
            seg = 1 + (r >> 1);
            unit = (bx - units) - r * units;
            sc_out = scan_slot(scan, kind, seg, units);
            mode = kind == 1 ? kSweepPhi : kSweepB;
        }
    } else {  // segments 1 .. P-1 from the combined start states
        seg = 1 + bx / units;
        unit = bx - (seg - 1) * units;
        sc_in = scan_slot(scan, 0, seg, units);
        mode = kSweepOut;
    }
    sweep_body<kBf16Out, kF32In>(&vmap, &omap, p, plan, n_max, ops, unit, 0, 0, sc_in, sc_out, mode, seg, P);
}

// S_{s+1} = Phi_s S_s + B_s for s = 1 .. P-2.  Stored transposed ([v][k]), with Phi stored the
// way the sweep stores a state (phiT[k'][k] = Phi[k][k']), this is X_{s+1} = X_s phiT + bT.  A
// block takes 8 rows v of one unit's state, a thread one column k; the rows of X stay in
// registers and shared memory, the segments follow one another.  Each Phi_s (64 KiB) is staged
// in shared memory by cp.async with all of it in flight at once: read straight from global
// memory inside the product, its loads left the kernel waiting on latency.
constexpr int kCombineRows = 8;
constexpr uint32_t CB_SMEM = kD * kD * 4 + kCombineRows * kD * 4 + 1024;

__global__ void __launch_bounds__(kD) prefill_scan_combine_kernel(float* __restrict__ scan, int units, int P) {
    extern __shared__ uint8_t smem_raw[];
    float* phs = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~static_cast<uintptr_t>(15));
    float* xs = phs + kD * kD;  // [kCombineRows][kD]
    const int blocks_per_unit = kD / kCombineRows;
    const int unit = blockIdx.x / blocks_per_unit, r0 = (blockIdx.x % blocks_per_unit) * kCombineRows;
    const int k = threadIdx.x;
    const size_t uo = (size_t)unit * kD * kD;
    float x[kCombineRows];
    const float* s1 = scan_slot(scan, 0, 1, units) + uo;
#pragma unroll
    for (int r = 0; r < kCombineRows; ++r) x[r] = s1[(r0 + r) * kD + k];
    const uint32_t phs_s = smem_u32(phs);
    for (int seg = 1; seg + 1 < P; ++seg) {
        const float* ph = scan_slot(scan, 1, seg, units) + uo;
        const float* bb = scan_slot(scan, 2, seg, units) + uo;
        // Phi_s -> shared memory: 4096 16-byte pieces, 32 per thread, consecutive per warp
#pragma unroll 8
        for (int e = k; e < kD * kD / 4; e += kD) cp_async16(phs_s + (uint32_t)e * 16, ph + 4 * e, 16);
        cp_async_commit();
        float acc[kCombineRows];
#pragma unroll
        for (int r = 0; r < kCombineRows; ++r) {
            acc[r] = bb[(r0 + r) * kD + k];
            xs[r * kD + k] = x[r];
        }
        cp_async_wait_all();
        __syncthreads();
#pragma unroll 2
        for (int kk = 0; kk < kD; kk += 4) {
            const float f0 = phs[kk * kD + k], f1 = phs[(kk + 1) * kD + k];
            const float f2 = phs[(kk + 2) * kD + k], f3 = phs[(kk + 3) * kD + k];
#pragma unroll
            for (int r = 0; r < kCombineRows; ++r) {
                const float4 xv = *reinterpret_cast<const float4*>(xs + r * kD + kk);
                acc[r] = fmaf(xv.x, f0, acc[r]);
                acc[r] = fmaf(xv.y, f1, acc[r]);
                acc[r] = fmaf(xv.z, f2, acc[r]);
                acc[r] = fmaf(xv.w, f3, acc[r]);
            }
        }
        float* nx = scan_slot(scan, 0, seg + 1, units) + uo;
#pragma unroll
        for (int r = 0; r < kCombineRows; ++r) {
            x[r] = acc[r];
            nx[(r0 + r) * kD + k] = acc[r];
        }
        __syncthreads();  // every thread is past its reads of phs and xs before they are rewritten
    }
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace

bool prefill_2p_supported(const PrefillArgs& p) { return p.M <= kTrack2p && p.N <= kMaxOrderN; }

// the segment scan's scratch is part of the workspace of up to kScanMaxN sequences of, on
// average, at least kScanMinChunks chunks
static bool scan_room(int64_t n_max, int32_t N) { return N <= kScanMaxN && n_max >= kScanMinChunks * N; }

size_t prefill_2p_workspace(int32_t T_tot, int32_t N, int32_t H) {
    if (N <= 0 || N > kMaxOrderN || T_tot < 0 || H <= 0) return 0;
    const int64_t n_max = max_chunks(T_tot, N);
    // plan, operand blocks, one fp32 state per (sequence, head) for the pipelined path, then
    // the segment scan's start / Phi / B states
    const size_t state = (size_t)kD * kD * 4;
    return ops_offset(n_max) + (size_t)n_max * (size_t)H * OP_BYTES + (size_t)N * H * state +
           (scan_room(n_max, N) ? (size_t)3 * kMaxSeg * N * H * state : 0);
}

namespace {

struct RawMaps {
    CUtensorMap q, k, g, v;
};

constexpr uint32_t PIPE_SMEM = PR_SMEM > SW_SMEM ? PR_SMEM : SW_SMEM;

// Segment count for the scan over sequences of about n chunks each and `units` (sequence, head)
// pairs, or 0 when it is not expected to beat one sweep of the sequence (the pipelined launches
// for one sequence, the plain sweep otherwise) by 10 %.  Cost in chunk-sweep times: the full
// prep (~2.3 sweep times per (chunk, head), spread over every SM), then launch 1 and launch 2,
// each as many waves of CTAs as it needs times the segment length.
int scan_segments(int64_t n, int units, int sms) {
    if (units <= 0 || sms <= 0) return 0;
    const double prep = 2.3 * (double)n * units / sms;
    double best = 0.9 * (double)n;
    int best_p = 0;
    for (int P = 3; P <= kMaxSeg; ++P) {
        const int64_t len = (n + P - 1) / P;
        const int64_t w1 = ((int64_t)units * (1 + 2 * (P - 2)) + sms - 1) / sms;
        const int64_t w2 = ((int64_t)units * (P - 1) + sms - 1) / sms;
        const double cost = prep + (double)(w1 + w2) * (double)len;
        if (cost < best) {
            best = cost;
            best_p = P;
        }
    }
    return best_p;
}

template <bool kBf16Out, bool kF32In>
void launch_2p(const RawMaps& m, const CUtensorMap& omap, const PrefillArgs& p, const int32_t* plan, int64_t n_max,
               uint8_t* ops, float* scratch, int sms, cudaStream_t s) {
    cudaFuncSetAttribute(prefill_prep_kernel<kBf16Out, kF32In>, cudaFuncAttributeMaxDynamicSharedMemorySize, PR_SMEM);
    cudaFuncSetAttribute(prefill_sweep_kernel<kBf16Out, kF32In>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         SW_SMEM);
    const int units = p.N * p.H;
    const int64_t H = p.H;
    auto prep = [&](int64_t c0, int64_t c1) {
        const int64_t items = (c1 - c0) * H;
        const unsigned grid = (unsigned)(items < (int64_t)sms ? items : sms);
        if (grid > 0)
            prefill_prep_kernel<kBf16Out, kF32In><<<grid, kThreads, PR_SMEM, s>>>(m.q, m.k, m.g, p, plan, n_max, ops,
                                                                                  c0, c1);
    };
    // Long sequences with few heads: swept as P segments at once when the cost model says so
    // (see scan_segments, with the mean sequence length), else pipelined (one sequence) or the
    // plain sweep below.
    const int P = scan_room(n_max, p.N) ? scan_segments(n_max / p.N, units, sms) : 0;
    if (P > 0) {
        float* scan = scratch + (size_t)p.N * p.H * kD * kD;
        cudaFuncSetAttribute(prefill_scan_kernel<kBf16Out, kF32In>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SW_SMEM);
        prep(0, n_max);
        prefill_scan_kernel<kBf16Out, kF32In><<<(unsigned)(units + 2 * units * (P - 2)), kSweepThreads, SW_SMEM,
                                                s>>>(m.v, omap, p, plan, n_max, ops, P, scan, units, 0);
        cudaFuncSetAttribute(prefill_scan_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, CB_SMEM);
        prefill_scan_combine_kernel<<<(unsigned)(units * (kD / kCombineRows)), kD, CB_SMEM, s>>>(scan, units, P);
        prefill_scan_kernel<kBf16Out, kF32In><<<(unsigned)(units * (P - 1)), kSweepThreads, SW_SMEM, s>>>(
            m.v, omap, p, plan, n_max, ops, P, scan, units, 1);
        return;
    }
    // One long sequence whose heads would leave most SMs idle in the sweep: chunk segments, a
    // short first one prepared on every SM, then each twice the one before, so that each is
    // prepared by the other SMs (at the launch's 96 registers, a little slower) while the sweep
    // runs through the previous one.
    const bool pipelined = p.N == 1 && units * 4 <= sms && n_max >= 256;
    if (!pipelined) {
        prep(0, n_max);
        prefill_sweep_kernel<kBf16Out, kF32In><<<units, kSweepThreads, SW_SMEM, s>>>(m.v, omap, p, plan, n_max, ops,
                                                                                     0, INT_MAX, nullptr, nullptr);
        return;
    }
    cudaFuncSetAttribute(prefill_pipe_kernel<kBf16Out, kF32In>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         PIPE_SMEM);
    int64_t b[16];
    int nb = 0;
    b[nb++] = 0;
    for (int64_t len = n_max / 32 > 0 ? n_max / 32 : 1; b[nb - 1] < n_max && nb < 15; len *= 2, ++nb)
        b[nb] = b[nb - 1] + len < n_max ? b[nb - 1] + len : n_max;
    b[nb - 1] = n_max;  // the last segment ends at the sequence's end
    prep(b[0], b[1]);
    for (int k = 0; k + 2 < nb; ++k)
        prefill_pipe_kernel<kBf16Out, kF32In><<<(unsigned)sms, kSweepThreads, PIPE_SMEM, s>>>(
            m.v, omap, m.q, m.k, m.g, p, plan, n_max, ops, scratch, units, (int)b[k], (int)b[k + 1], b[k + 1],
            b[k + 2]);
    prefill_sweep_kernel<kBf16Out, kF32In><<<units, kSweepThreads, SW_SMEM, s>>>(m.v, omap, p, plan, n_max, ops,
                                                                                 (int)b[nb - 2], INT_MAX, scratch,
                                                                                 nullptr);
}

}  // namespace

kda_status launch_prefill_2p(const PrefillArgs& p, bool bf16_in, bool bf16_out, void* workspace, cudaStream_t s) {
    const int64_t n_max = max_chunks(p.T_tot, p.N);
    int32_t* plan = static_cast<int32_t*>(workspace);
    uint8_t* ops = static_cast<uint8_t*>(workspace) + ops_offset(n_max);
    // bf16 activations as 2-D tensors [T_tot rows][H * 128]: the prep loads a (chunk, head)'s
    // raw q, k, g as one 128-channel x 64-token box each (row-major, unswizzled); the sweep loads
    // its V as two 64-channel x 64-token boxes, 128-byte swizzled (the MN-major MMA operand
    // layout).  Rows past T_tot read as zero.
    RawMaps maps;
    memset(&maps, 0, sizeof(maps));
    if (p.T_tot > 0 && bf16_in) {
        PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
        if (enc == nullptr) return KDA_ERR_CUDA;
        const cuuint64_t dims[2] = {(cuuint64_t)p.H * kD, (cuuint64_t)p.T_tot};
        const cuuint64_t strides[1] = {(cuuint64_t)p.H * kD * 2};
        const cuuint32_t estr[2] = {1, 1};
        const cuuint32_t box_raw[2] = {128, 64};
        const void* raw[3] = {p.q, p.k, p.gate_raw};
        CUtensorMap* dst[3] = {&maps.q, &maps.k, &maps.g};
        for (int i = 0; i < 3; ++i)
            if (enc(dst[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(raw[i]), dims, strides, box_raw,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
                return KDA_ERR_CUDA;
        const cuuint32_t box[2] = {64, 64};
        if (enc(&maps.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.v), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return KDA_ERR_CUDA;
    }
    // out as [T_tot rows][H * 128] bf16: a full chunk's outputs leave as one 128 x 64 box
    CUtensorMap omap;
    memset(&omap, 0, sizeof(omap));
    if (p.T_tot > 0 && bf16_out) {
        PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
        if (enc == nullptr) return KDA_ERR_CUDA;
        const cuuint64_t dims[2] = {(cuuint64_t)p.H * kD, (cuuint64_t)p.T_tot};
        const cuuint64_t strides[1] = {(cuuint64_t)p.H * kD * 2};
        const cuuint32_t box[2] = {128, 64};
        const cuuint32_t estr[2] = {1, 1};
        if (enc(&omap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.out, dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return KDA_ERR_CUDA;
    }
    prefill_plan_kernel<<<1, kPlanThreads, 0, s>>>(p.cu_seqlens, p.N, p.T_tot, n_max, plan);
    const int sms = sm_count() > 0 ? sm_count() : 1;
    float* scratch = reinterpret_cast<float*>(ops + (size_t)n_max * (size_t)p.H * OP_BYTES);
    if (bf16_in && bf16_out)
        launch_2p<true, false>(maps, omap, p, plan, n_max, ops, scratch, sms, s);
    else if (bf16_in)
        launch_2p<false, false>(maps, omap, p, plan, n_max, ops, scratch, sms, s);
    else if (bf16_out)
        launch_2p<true, true>(maps, omap, p, plan, n_max, ops, scratch, sms, s);
    else
        launch_2p<false, true>(maps, omap, p, plan, n_max, ops, scratch, sms, s);
    return launch_status();
}

}  // namespace kda
