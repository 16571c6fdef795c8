// Paged MLA decode on sm_103a: tcgen05 tensor-core contractions over a
// paged latent cache, with online softmax and split-KV partials.
//
// What is computed (absorbed MLA decode, "sabi-mla-vllm" README intro and
// "What the plugin does"; multi-token causal verify from "qwen-mla-vllm"
// README "Speculative decoding (MTP)"; LSE output and the (0, -inf) rule from
// vLLM PR #55543 commit 5.1-5.4):
//   s_j = scale * (q_lat . c_j + q_pe . k_pe_j),  out = softmax(s) . c,
//   lse = ln sum_j exp(s_j), over the tokens each query row may see.
//
// Two decode kernels share the work split, the split-KV partials and the
// merge:
//   mla_decode_fold_kernel  64-token tiles folded into two 288-value halves
//                           (see "folded tiles" below): every pool whose page
//                           size is a multiple of 8 rows, except fp8_ds_mla
//                           pools at up to 32 or above 64 query rows.
//   mla_decode_kernel       128-token tiles whose 576 dims are split over the
//                           two CTAs of a cluster: those fp8 pools, and pages
//                           that are not a multiple of 8 rows (load/convert
//                           warps read them).
//
// Work split ("stream-K" over tiles). The tiles of all requests are
// concatenated and the workers (a CTA, or a cluster of two) each take an
// equal contiguous range of the cost (a request boundary counts as a few
// tiles), so every SM streams about the same number of cache bytes whatever
// the request lengths. The tiles of one request inside a range form a
// segment; a segment covering its whole request writes the final output,
// otherwise an fp32 partial (out, lse) that a second kernel merges. Query
// rows (query token x head) are processed in groups of at most 64 (NP = 16,
// 32 or 64, padded); gridDim.y covers more.
//
// Cluster kernel. Two CTAs per tile (a cluster of 2 on neighbouring SMs)
// split the 576 cached dims: CTA r holds latent dims [256r, 256r+256) and
// rope dims [512+32r, 512+32r+32), i.e. 72 KB of each 128-token tile, so two
// or more tiles fit in shared memory and loads overlap compute. Per tile:
//   S_r^T[128 tok, NP] = C_r[128, 288] . Q_r^T        (UMMA M=128, into TMEM)
//   S = S_0 + S_1       (each CTA sends its partial to the other through
//                        distributed shared memory)
//   P = exp2(S*scale*log2e - m)   (bf16, identical in both CTAs)
//   O_r^T[256, NP] += C_r[128, 0:256]^T . P^T          (2 UMMAs of M=128)
// C stays in shared memory in the 128-byte-swizzled layout that is the K-major
// A operand of the first product and the MN-major A operand of the second.
// All query rows share one read of the cache (the pages' point that a verify
// step must read the latent once per request).
//
// Warp roles of the cluster kernel's CTAs:
//   warp 0      : TMEM allocation; lane 0 issues the S = C.Q^T MMAs
//   warp 1      : TMA producer (page_size % 8 == 0)
//   warp 2      : tile-range scan at start
//   warp 3      : lane 0 issues the O += C^T.P MMAs
//   warps 4..7  : softmax, P, output epilogue (thread t <-> token t <-> TMEM lane t)
//   warps 8..11 : fp8 pools: expand the e4m3 codes that the TMA producer
//                 landed in a tile's pair slots into bf16 in place; odd page
//                 sizes: load/convert producers that read the pool directly
//
// Online softmax with a lazily raised maximum: m moves only when a score
// exceeds it by more than 2^8 (log2 units), so P <= 256 and rescaling O is
// rare; l is kept per thread and reduced once per segment.
#include <climits>
#include <cstddef>

#include "launch.cuh"
#include "mla_common.cuh"

namespace mla {

// Pipeline timeline for development builds (-DMLA_TRACE): %globaltimer at
// hand-off points for the first 8 CTAs and 64 tiles, read back by the host
// through mla_trace_dump(). Compiles to nothing otherwise.
enum TraceEvent : int {
    kTrProdStart = 0, kTrProdIssued, kTrSPair0, kTrSAllIn, kTrPvIssue, kTrSmSFull, kTrSmXFull, kTrSmPArrive,
    kTrSIssued = 8, kTrSmTmemLd, kTrSmXFree, kTrSmSent, kTrSmMath, kTrSmBarOr, kTrSmExp, kTrSmPStore, kTrPvIssued,
    kTrSmXRead, kTrSmExpLoop, kTrEpiStart, kTrEpiRed, kTrEpiStored, kTrEpiEnd, kTrEpiHalf,
    kTrSKb1 = 24, kTrSKb2, kTrSKb3, kTrSRope, kTrProd1Start, kTrProd1Done, kTrProd0Done, kTrSmRescaled,
    kTrEvents = 32
};
#ifdef MLA_TRACE
__device__ unsigned long long g_trace[8][64][kTrEvents];
#define MLA_TRACE_POINT(i, e)                                                                     \
    do {                                                                                          \
        if (blockIdx.y == 0 && blockIdx.x < 8 && (i) < 64) g_trace[blockIdx.x][(i)][(e)] = globaltimer_ns(); \
    } while (0)
// whole-kernel points per CTA (row group 0): entry, setup done, softmax
// done, exit; and entry/exit of each merge block
__device__ unsigned long long g_ktrace[512][4];
// per CTA (row group 0) and tile: when the softmax handed P to the PV issuer
__device__ unsigned long long g_ttrace[512][1024];
__device__ unsigned int g_ksm[512][4];  // smid, tiles, segments
__device__ unsigned long long g_mtrace[512][2];
#define MLA_KTRACE(e)                                                                  \
    do {                                                                               \
        if (blockIdx.y == 0 && blockIdx.x < 512) g_ktrace[blockIdx.x][(e)] = globaltimer_ns(); \
    } while (0)
#define MLA_TTRACE(i)                                                                            \
    do {                                                                                         \
        if (blockIdx.y == 0 && blockIdx.x < 512 && (i) < 1024) g_ttrace[blockIdx.x][(i)] = globaltimer_ns(); \
    } while (0)
#define MLA_KSM(k, v)                                             \
    do {                                                          \
        if (blockIdx.y == 0 && blockIdx.x < 512) g_ksm[blockIdx.x][(k)] = (v); \
    } while (0)
#define MLA_MTRACE(e)                                                                   \
    do {                                                                                \
        if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.x < 512) g_mtrace[blockIdx.x][(e)] = globaltimer_ns(); \
    } while (0)
#else
#define MLA_TRACE_POINT(i, e) \
    do {                      \
    } while (0)
#define MLA_KTRACE(e) \
    do {              \
    } while (0)
#define MLA_MTRACE(e) \
    do {              \
    } while (0)
#define MLA_TTRACE(i) \
    do {              \
    } while (0)
#define MLA_KSM(k, v) \
    do {              \
    } while (0)
#endif

constexpr float kRescaleThreshold = 8.0f;  // log2 units
// fp8 rows widened to f16: |code| <= 448, so a block scale up to this keeps
// every widened value (and its product with the scale) within the f16 range
constexpr float kMaxF16Scale = 146.0f;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr int kPrefetchTiles = 2;          // L2 lookahead of the load/convert producers
constexpr int kRawSlots = 3;               // fp8 tiles in flight between TMA and the expand warps

template <int NP, bool LSU>
struct Cfg {
    static_assert(NP == 16 || NP == 32 || NP == 64, "NP");
    static constexpr int kPairBytes = 2 * 128 * 128;  // 2 x (64 dims x 128 tokens), 128-B swizzled
    static constexpr int kRopeBytes = 128 * 64;       // 32 rope dims x 128 tokens, 64-B swizzled
    // Pair slots (2 per tile). Pair pk of every tile is freed by PV issuer pk;
    // the load/convert warps of pair pk order their refills only by their own
    // earlier waits, which with an odd ring would see the other issuer's
    // progress only and could not prove that the slot's fill before last was
    // freed (a parity wait cannot tell the two apart) while issuer pk runs
    // behind. With an even ring a slot always holds the same pair. The single
    // TMA producer waits on both pairs, so 5 slots are sound there.
    static constexpr int kRL = (NP == 64 || LSU) ? 4 : 5;
    static constexpr int kRR = (NP == 16) ? 3 : (NP == 32 ? 2 : 1);  // rope slots (1 per tile; freed right after S)
    static constexpr int kQBytes = NP * (4 * 128 + 64);
    // 32 and 64 query rows: the two CTAs split the softmax columns, each owning
    // kNH of them; 16 rows: both run the whole softmax
    static constexpr bool kSplit = NP >= 32;
    static constexpr int kNH = kSplit ? NP / 2 : NP;
    static constexpr int kXBytes = 128 * kNH * 4;     // the peer's partial S of this CTA's columns
    static constexpr int kPBufs = (NP == 64) ? 1 : 2; // P (bf16) buffers
    static constexpr int kPBytes = 128 * NP * 2;
    static constexpr int kOffRope = kRL * kPairBytes;
    static constexpr int kOffQ = kOffRope + kRR * kRopeBytes;
    static constexpr int kOffX = (kOffQ + kQBytes + 1023) / 1024 * 1024;
    static constexpr int kOffP = kOffX + kXBytes;
    // Send buffer of the score exchange: the partial S of the peer's columns
    // is staged here and pushed to the peer by one bulk copy. At 32 rows it is
    // the tile's own P buffer (the same 8 KB, idle until P is written), which
    // pays for the fifth pair slot.
    static constexpr bool kSendInP = (NP == 32);
    static_assert(!kSendInP || kXBytes == kPBytes, "send staging in the P buffer");
    static constexpr int kOffSend = kOffP + kPBufs * kPBytes;
    static constexpr int kOffCtrl = kOffSend + (kSendInP ? 0 : kXBytes);
    static constexpr int kSmemBytes = kOffCtrl + 3584 + 1024;  // + control block, alignment slack
    // TMEM: two O accumulators of 2 x NP columns (one per alternating
    // segment, so a finished segment drains while the next accumulates),
    // then two S buffers of NP columns
    static constexpr int kTmemCols = NP == 16 ? 128 : NP == 32 ? 256 : 512;
    static constexpr int kColS = 4 * NP;
    // P: NP / kNH column blocks of [128 tokens][kNH bf16], MN-major, swizzled by
    // the block width, so each CTA's softmax columns are one contiguous block
    static constexpr uint32_t kPSwizzle = kNH == 16 ? kSw32 : kSw64;
    static constexpr int kPBlockBytes = 128 * kNH * 2;
    static_assert(kSmemBytes <= 232448, "shared memory");
    static_assert(kTmemCols >= 32, "tmem");
};

struct Ctrl {
    uint64_t pair_full[5], pair_empty[5];
    uint64_t rope_full[3], rope_empty[3];
    uint64_t s_full[2], s_free[2], o_done[2], q_full;
    // tile t's P hand-off to the two PV issuers is p_full[t & 1]: the softmax
    // may hand over tile t + 1 as soon as PV(t - 1) is done, which can be
    // before a slow issuer has begun to wait for tile t, and one barrier would
    // then complete a phase past that issuer, whose parity wait could never
    // end; tile t + 2's hand-off follows PV(t) of both issuers
    uint64_t p_full[2];
    uint64_t xfull;          // the peer's partial S landed (st.async transactions + 1 local arrive)
    uint64_t xfree;          // the peer has read this CTA's last partial S (1 remote arrive)
    uint64_t raw_full[3];    // fp8: a tile's codes and scales landed in its pair slots
    uint32_t tmem_base;
    int abort;
    int t_begin, t_end, b0, j0;
    int colvis[64];                  // uniform verify length: query row -> trailing tokens it may not see
    alignas(16) float m[64];         // running max per row (log2 units); read as float4
    alignas(16) float alpha[64];
    alignas(16) float red[4][64];
    alignas(16) float dlt[2][64];    // row sums of a finished segment, by segment parity
    float dm[64];                    // and the row maxima of this CTA's columns
    alignas(16) float palpha[2][32]; // the peer's rescale factors for its columns, by P buffer
    alignas(16) int pflag[2][4];     // and whether it rescaled this tile
    uint64_t pin[2];                 // the peer's P block and message landed (by P buffer)
    uint64_t rp_free[2];             // the peer's P buffer may be written (its PV is done)
    uint64_t dfull[2];               // the peer's row sums of a segment landed (by parity)
};
static_assert(sizeof(Ctrl) <= 3584, "control block");
static_assert(offsetof(Ctrl, m) % 16 == 0 && offsetof(Ctrl, alpha) % 16 == 0, "vector loads of m / alpha");

__device__ __forceinline__ int swz_p(int row, uint32_t mode) {
    return mode == kSw128 ? (row & 7) : mode == kSw64 ? ((row >> 1) & 3) : ((row >> 2) & 1);
}

// Walks the tiles (1 << SH tokens each) of consecutive requests.
template <int SH>
struct TileItT {
    int b, j, tiles, T;
    __device__ __forceinline__ void init(const int32_t* sl, int b0, int j0) {
        b = b0;
        j = j0;
        T = max(__ldg(sl + b), 0);
        tiles = (T + (1 << SH) - 1) >> SH;
    }
    __device__ __forceinline__ void next(const int32_t* sl, int B) {
        if (++j >= tiles) {
            j = 0;
            do {
                ++b;
                if (b >= B) { T = 0; tiles = 1; break; }
                T = max(__ldg(sl + b), 0);
                tiles = (T + (1 << SH) - 1) >> SH;
            } while (tiles == 0);
        }
    }
};
using TileIt = TileItT<7>;

// Query rows of request b: the first row of its verify step and the step's
// length in tokens (Qt for every request unless per-request lengths are given),
// and how many of its rows fall in row group gy (0 .. 64). Per-request prefix
// sums are clamped to [0, total_q], so whatever they hold no row past the
// query, output and LSE buffers is touched (a request whose sums run past
// total_q keeps its tokens below it).
__device__ __forceinline__ int cu_clamped(const DecodeParams& p, int b) {
    return min(max(__ldg(p.cu_q + b), 0), p.total_q);
}
__device__ __forceinline__ int64_t req_row0(const DecodeParams& p, int b) {
    return p.cu_q ? static_cast<int64_t>(cu_clamped(p, b)) * p.Hq : static_cast<int64_t>(b) * p.HQ;
}
__device__ __forceinline__ int req_qt(const DecodeParams& p, int b) {
    return p.cu_q ? cu_clamped(p, b + 1) - cu_clamped(p, b) : p.Qt;
}
__device__ __forceinline__ int req_rows_in_group(const DecodeParams& p, int b, int gy) {
    return min(64, max(0, req_qt(p, b) * p.Hq - gy * 64));
}

// L2 prefetch of what the first tiles of request b read besides the cache:
// its query rows of row group gy and its block-table row (whole 16-byte
// units inside the row only).
__device__ __forceinline__ void prefetch_request(const DecodeParams& p, int b, int gy) {
    const int HQg = req_rows_in_group(p, b, gy);
    const int64_t row0 = req_row0(p, b) + gy * 64;
    if (HQg > 0) {
        prefetch_l2_bulk(p.q_lat + row0 * p.lat_dim, static_cast<uint32_t>(HQg * p.lat_dim * 2));
        prefetch_l2_bulk(p.q_pe + row0 * p.rope_dim, static_cast<uint32_t>(HQg * p.rope_dim * 2));
    }
    const int T = max(__ldg(p.seq_lens + b), 0);
    const int64_t pages = min((static_cast<int64_t>(T) + p.page_size - 1) / p.page_size, p.bt_stride);
    uintptr_t a0 = reinterpret_cast<uintptr_t>(p.block_table + static_cast<int64_t>(b) * p.bt_stride);
    uintptr_t a1 = a0 + static_cast<uintptr_t>(pages) * 4;
    a0 = (a0 + 15) & ~static_cast<uintptr_t>(15);
    a1 &= ~static_cast<uintptr_t>(15);
    if (a1 > a0) {
        const uintptr_t n = a1 - a0;
        prefetch_l2_bulk(reinterpret_cast<const void*>(a0), static_cast<uint32_t>(n < (1u << 20) ? n : (1u << 20)));
    }
}

// Work split. Tiles of all requests in order form one sequence; a non-empty
// request also carries wseg units of cost before its first tile (what a
// request boundary costs a cluster: the next request's queries, the drain of
// the previous output). Cluster g of G takes the tiles whose cost coordinate
// lies in [g*C/G, (g+1)*C/G), C the total cost. Both functions are called by
// a whole warp and return the same value in every lane.

// Total tiles and total cost over all requests.
template <int SH>
__device__ __forceinline__ void work_totals(const int32_t* sl, int B, int wseg, int lane, long long& tiles,
                                            long long& cost) {
    long long t = 0, c = 0;
    for (int base = 0; base < B; base += 32) {
        const int b = base + lane;
        const int tl = b < B ? (max(__ldg(sl + b), 0) + (1 << SH) - 1) >> SH : 0;
        int st = tl, sc = tl > 0 ? tl + wseg : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            st += __shfl_xor_sync(0xffffffffu, st, o);
            sc += __shfl_xor_sync(0xffffffffu, sc, o);
        }
        t += st;
        c += sc;
    }
    tiles = t;
    cost = c;
}

// Number of tiles whose cost coordinate is below x.
template <int SH>
__device__ __forceinline__ long long tiles_before_cost(const int32_t* sl, int B, int wseg, long long x, int lane) {
    long long acc_c = 0, acc_t = 0;
    for (int base = 0; base < B; base += 32) {
        const int b = base + lane;
        const int tl = b < B ? (max(__ldg(sl + b), 0) + (1 << SH) - 1) >> SH : 0;
        const int cb = tl > 0 ? tl + wseg : 0;
        int ic = cb, it = tl;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int vc = __shfl_up_sync(0xffffffffu, ic, o);
            const int vt = __shfl_up_sync(0xffffffffu, it, o);
            if (lane >= o) {
                ic += vc;
                it += vt;
            }
        }
        const unsigned hit = __ballot_sync(0xffffffffu, b < B && acc_c + ic > x);
        if (hit) {
            const int L = __ffs(hit) - 1;
            const long long cs = acc_c + __shfl_sync(0xffffffffu, ic, L) - __shfl_sync(0xffffffffu, cb, L);
            const long long ts = acc_t + __shfl_sync(0xffffffffu, it, L) - __shfl_sync(0xffffffffu, tl, L);
            const long long in = x - cs - wseg;  // tiles of request L below x
            return ts + (in > 0 ? in : 0);
        }
        acc_c += __shfl_sync(0xffffffffu, ic, 31);
        acc_t += __shfl_sync(0xffffffffu, it, 31);
    }
    return acc_t;
}

// Tile range [tb, te) of worker g of G and the request / tile it starts at.
// Called by a whole warp; every lane returns the same values.
struct TileRange {
    int tb, te, b0, j0;
};
template <int SH>
__device__ __forceinline__ TileRange scan_range(const DecodeParams& p, int g, int G, int lane) {
    long long total = 0, cost = 0;
    work_totals<SH>(p.seq_lens, p.B, p.wseg, lane, total, cost);
    const int tb = static_cast<int>(tiles_before_cost<SH>(p.seq_lens, p.B, p.wseg, g * cost / G, lane));
    const int te = static_cast<int>(tiles_before_cost<SH>(p.seq_lens, p.B, p.wseg, (g + 1) * cost / G, lane));
    int b0 = 0, j0 = 0;
    long long acc = 0;
    for (int base = 0; base < p.B; base += 32) {
        const int b = base + lane;
        const int tl = b < p.B ? (max(__ldg(p.seq_lens + b), 0) + (1 << SH) - 1) >> SH : 0;
        int incl = tl;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        const long long gi = acc + incl;
        const unsigned hit = __ballot_sync(0xffffffffu, b < p.B && tl > 0 && gi > tb);
        if (hit) {
            const int L = __ffs(hit) - 1;
            const long long gl = __shfl_sync(0xffffffffu, gi, L);
            const int tll = __shfl_sync(0xffffffffu, tl, L);
            b0 = base + L;
            j0 = static_cast<int>(tb - (gl - tll));
            break;
        }
        acc += __shfl_sync(0xffffffffu, incl, 31);
    }
    TileRange r;
    r.tb = tb;
    r.te = te;
    r.b0 = b0;
    r.j0 = j0;
    return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int NP>
__device__ __forceinline__ void tmem_ld_np(uint32_t taddr, uint32_t (&r)[NP]) {
    if constexpr (NP == 8) tmem_ld_x8(taddr, r);
    else if constexpr (NP == 16) tmem_ld_x16(taddr, r);
    else if constexpr (NP == 32) tmem_ld_x32(taddr, r);
    else tmem_ld_x64(taddr, r);
}

// Wait sites, recorded with the first failure (workspace header words 1..3:
// site, tile index within the CTA's range, linear block index).
enum WaitSite : int {
    kSiteQFull = 1, kSiteSFree, kSitePairFull, kSiteRopeFull, kSitePFull, kSiteTmaPairEmpty, kSiteTmaRopeEmpty,
    kSiteLsuPairEmpty, kSiteLsuRopeEmpty, kSiteSFull, kSiteXFree, kSiteXFull, kSiteOEpi, kSiteORescale, kSiteOPbuf,
    kSiteOFinal, kSiteRawFull, kSiteDFull, kSitePIn, kSiteRpFree
};

// This CTA's status record; zeroed by the CTA itself at launch and folded
// into the workspace header by the merge step.
__device__ __forceinline__ int* status_rec(const DecodeParams& p) {
    return p.rec + static_cast<int64_t>(blockIdx.y * gridDim.x + blockIdx.x) * kStatusRecWords;
}

template <class CT>
__device__ __forceinline__ void fail(const DecodeParams& p, CT* ctrl, int code, int site = 0, int tile = 0) {
    int* r = status_rec(p);
    atomicOr(r, code);
    if (site && atomicCAS(r + 1, 0, site) == 0) r[2] = tile;
    ctrl->abort = 1;
}

// Every softmax thread waits, then the 128 threads agree on the outcome, so a
// timeout seen by some of them cannot strand the rest at a named barrier.
// When a role leaves its loop on a failed wait it records where it was
// waiting: record word 4 + role = (site << 24) | tile.
enum Role : int { kRoleS = 0, kRolePV, kRoleSoftmax, kRoleTma, kRoleLsu0 };

__device__ __forceinline__ void report(const DecodeParams& p, int role, int site, int idx) {
    status_rec(p)[4 + role] = (site << 24) | (idx & 0xFFFFFF);
}

// Softmax-group wait. A thread whose wait fails raises the abort flag and
// carries on (its results no longer matter); the group leaves its tile loop
// together after the tile's last barrier, where every thread reads the flag.
template <class CT>
__device__ __forceinline__ bool group_wait(uint64_t* bar, uint32_t parity, const DecodeParams& p, CT* ctrl,
                                           int site, int tile, bool cluster_scope = false) {
    const bool ok = cluster_scope ? mbar_wait_cluster(bar, parity, &ctrl->abort) : mbar_wait(bar, parity, &ctrl->abort);
    if (!ok) {
        fail(p, ctrl, kErrWaitTimeout, site, tile);
        report(p, kRoleSoftmax, site, tile);
    }
    return ok;
}

// 64-bit slot of token `tok` of the request whose block-table row is `btr`.
__device__ __forceinline__ int64_t token_slot(const DecodeParams& p, const int32_t* btr, int tok, bool& bad) {
    const int pi = tok / p.page_size;
    // a page index past the block-table row (a sequence longer than the table)
    // counts as an entry outside the pool
    const int64_t page = pi < p.bt_stride ? __ldg(btr + pi) : -1;
    const int64_t ps = p.page_size;
    if (page < 0 || (page + 1) * ps > p.num_slots) {
        bad = true;
        return tok % p.page_size;  // page 0: in bounds, flagged
    }
    return page * ps + tok % p.page_size;
}

// Ask L2 for the cache rows of tile t, one bulk prefetch per run of tokens
// sharing a page (their rows are contiguous); runs alternate between the two
// CTAs of the cluster.
__device__ __forceinline__ void prefetch_tile(const DecodeParams& p, const TileIt& t, int row_bytes, int rank) {
    const int valid = min(kTile, t.T - t.j * kTile);
    const int32_t* btr = p.block_table + static_cast<int64_t>(t.b) * p.bt_stride;
    bool bad = false;
    int tok = t.j * kTile, k = 0;
    const int end = tok + valid;
    while (tok < end) {
        const int run = min(end, (tok / p.page_size + 1) * p.page_size) - tok;
        if ((k++ & 1) == rank) {
            const int64_t slot = token_slot(p, btr, tok, bad);
            if (!bad) prefetch_l2_bulk(p.cache + slot * row_bytes, static_cast<uint32_t>(run * row_bytes));
        }
        tok += run;
    }
}

// Threads per CTA: 8 warps, plus 4 load/convert or expand warps.
template <bool LSU, int KIND>
constexpr int decode_threads() { return (LSU || KIND == 1) ? 384 : 256; }

template <int NP, bool LSU, int KIND>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(decode_threads<LSU, KIND>(), 1)
    mla_decode_kernel(const __grid_constant__ DecodeMaps maps, const DecodeParams p) {
    const CUtensorMap& tmap_lat = maps.lat;
    const CUtensorMap& tmap_rope = maps.rope;
    using C = Cfg<NP, LSU>;
    extern __shared__ uint8_t smem_raw[];
    // align by offset from the shared array so every derived pointer stays a
    // shared-space pointer (ld/st.shared rather than generic accesses)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* pair_ring = smem;
    uint8_t* rope_ring = smem + C::kOffRope;
    uint8_t* qs = smem + C::kOffQ;
    uint8_t* xbuf = smem + C::kOffX;
    uint8_t* pbufs = smem + C::kOffP;
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + C::kOffCtrl);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = static_cast<int>(cluster_ctarank());
    const int g = blockIdx.x >> 1, G = gridDim.x >> 1, gy = blockIdx.y;
    if (threadIdx.x == 0) MLA_KTRACE(0);

    if (threadIdx.x == 0) {
        // TMA: one expect_tx arrival per fill; load/convert warps: one arrival per
        // warp that writes part of the fill (2 per pair, 4 per rope slot)
        // pair fill arrivals: TMA (1, with bytes), load/convert warps (2 per
        // pair), expand warps (4 per pair)
        constexpr int kPairArrivals = LSU ? 2 : (KIND == 1 ? 4 : 1);
        for (int i = 0; i < C::kRL; ++i) { mbar_init(&ctrl->pair_full[i], kPairArrivals); mbar_init(&ctrl->pair_empty[i], 1); }
        for (int i = 0; i < kRawSlots; ++i) mbar_init(&ctrl->raw_full[i], 1);
        for (int i = 0; i < C::kRR; ++i) { mbar_init(&ctrl->rope_full[i], LSU ? 4 : 1); mbar_init(&ctrl->rope_empty[i], 1); }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctrl->s_full[i], 1);
            mbar_init(&ctrl->s_free[i], 1);
            mbar_init(&ctrl->o_done[i], 2);  // one commit per PV issuer
        }
        mbar_init(&ctrl->p_full[0], 1);
        mbar_init(&ctrl->p_full[1], 1);
        mbar_init(&ctrl->q_full, 1);
        mbar_init(&ctrl->xfull, 1);
        mbar_init(&ctrl->xfree, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctrl->pin[i], 1);
            mbar_init(&ctrl->rp_free[i], 1);
            mbar_init(&ctrl->dfull[i], 1);
        }
        ctrl->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1 && lane == 0) {
        if (!LSU) {
            prefetch_tensormap(&tmap_lat);
            prefetch_tensormap(&tmap_rope);
        }
        prefetch_tensormap(&maps.q);
        prefetch_tensormap(&maps.qpe);
    }
    // everything above touches only this CTA; the previous kernel in the
    // stream may still be writing the inputs or reading the workspace
    griddep_wait();
    if (threadIdx.x == 0) {
        int4* r = reinterpret_cast<int4*>(status_rec(p));
#pragma unroll
        for (int k = 0; k < kStatusRecWords / 4; ++k) r[k] = make_int4(0, 0, 0, 0);
    }
    if (warp == 0) {
        tmem_alloc(&ctrl->tmem_base, C::kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    if (warp == 2) {
        // this cluster's tile range (cost-weighted split) and where it starts
        const TileRange r = scan_range<7>(p, g, G, lane);
        if (lane == 0) {
            ctrl->t_begin = r.tb;
            ctrl->t_end = r.te;
            ctrl->b0 = r.b0;
            ctrl->j0 = r.j0;
        }
    }
    if (threadIdx.x >= 128 && threadIdx.x < 128 + 64) {
        const int c = threadIdx.x - 128;
        const int r = gy * 64 + c;
        ctrl->colvis[c] = (r < p.HQ) ? (p.Qt - 1 - r / p.Hq) : (INT_MAX / 2);
        ctrl->m[c] = -INFINITY;
    }
    __syncthreads();
    cluster_sync_all();  // the peer's barriers exist before any remote arrive
    if (threadIdx.x == 0) {
        MLA_KTRACE(1);
#ifdef MLA_TRACE
        unsigned sm;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
        MLA_KSM(0, sm);
        MLA_KSM(1, ctrl->t_end - ctrl->t_begin);
#endif
        griddep_launch_dependents();  // the merge grid may be scheduled as CTAs retire
    }
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    const int ntiles = ctrl->t_end - ctrl->t_begin;
    if (ntiles == 0 && ctrl->j0 > 0 && rank == 0 && threadIdx.x >= 128 && threadIdx.x < 192) {
        // An empty range strictly inside request b0 (more clusters than
        // tiles): the merge of b0 counts this cluster's slot, so mark it empty.
        const int64_t pslot = static_cast<int64_t>(gy) * p.SPG + g + ctrl->b0;
        p.part_lse[pslot * 64 + (threadIdx.x - 128)] = -INFINITY;
    }

    if (ntiles > 0) {
        if (warp == 0 && lane == 0) {
            // -------------------------------------------------- S issuer
            // S(i) into TMEM buffer i%2 as soon as tile i is in shared memory
            // and the softmax has read S(i-2) from that buffer.
            TileIt it;
            it.init(p.seq_lens, ctrl->b0, ctrl->j0);
            const uint32_t idS = idesc_bf16(128, NP, false, false);
            const uint64_t dq = smem_desc(smem_u32(qs), 16, 1024, kSw128);
            const uint64_t dqr = smem_desc(smem_u32(qs) + 4 * NP * 128, 16, 512, kSw64);
            int seg = 0;
            for (int i = 0; i < ntiles; ++i) {
                if (i == 0 || it.j == 0) {
                    if (!mbar_wait(&ctrl->q_full, seg & 1, &ctrl->abort)) {
                        fail(p, ctrl, kErrWaitTimeout, kSiteQFull, i);
                        report(p, kRoleS, kSiteQFull, i);
                        break;
                    }
                    ++seg;
                }
                if (i >= 2 && !mbar_wait(&ctrl->s_free[i & 1], ((i - 2) >> 1) & 1, &ctrl->abort)) {
                    fail(p, ctrl, kErrWaitTimeout, kSiteSFree, i);
                    report(p, kRoleS, kSiteSFree, i);
                    break;
                }
                const uint32_t tS = tmem + C::kColS + (i & 1) * NP;
                bool ok = true;
                int site = kSitePairFull;
                for (int pp = 0; pp < 2 && ok; ++pp) {
                    const int u = 2 * i + pp, slot = u % C::kRL;
                    if (!mbar_wait(&ctrl->pair_full[slot], (u / C::kRL) & 1, &ctrl->abort)) { ok = false; break; }
                    tc_fence_after();
                    if (pp == 0) MLA_TRACE_POINT(i, kTrSPair0);
                    const uint64_t da = smem_desc(smem_u32(pair_ring + slot * C::kPairBytes), 16, 1024, kSw128);
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            umma_bf16(tS, da + ((c * 16384 + kk * 32) >> 4), dq + (((2 * pp + c) * NP * 128 + kk * 32) >> 4),
                                      idS, (pp | c | kk) != 0);
                }
                const int rr = i % C::kRR;
                if (ok && !mbar_wait(&ctrl->rope_full[rr], (i / C::kRR) & 1, &ctrl->abort)) {
                    ok = false;
                    site = kSiteRopeFull;
                }
                if (!ok) {
                    fail(p, ctrl, kErrWaitTimeout, site, i);
                    report(p, kRoleS, site, i);
                    break;
                }
                tc_fence_after();
                MLA_TRACE_POINT(i, kTrSAllIn);
                const uint64_t dr = smem_desc(smem_u32(rope_ring + rr * C::kRopeBytes), 16, 512, kSw64);
                umma_bf16(tS, dr, dqr, idS, 1u);
                umma_bf16(tS, dr + 2, dqr + 2, idS, 1u);
                umma_commit(&ctrl->s_full[i & 1]);
                umma_commit(&ctrl->rope_empty[rr]);
                MLA_TRACE_POINT(i, kTrSIssued);
                it.next(p.seq_lens, p.B);
            }
        } else if ((warp == 3 || warp == 2) && lane == 0) {
            // ------------------------------------------------- PV issuers
            // warp 3 issues the first 128 latent dims of this CTA (O half 0), warp
            // 2 the second: independent accumulators, so two threads halve the
            // issue time and the pair slots come free sooner
            const int mt = warp == 3 ? 0 : 1;
            TileIt it;
            it.init(p.seq_lens, ctrl->b0, ctrl->j0);
            const uint32_t idPV = idesc_bf16(128, NP, true, true);
            constexpr uint32_t p_sbo = 8 * C::kNH * 2;
            int seg = -1;
            for (int i = 0; i < ntiles; ++i) {
                const bool new_seg = (i == 0) || (it.j == 0);
                if (new_seg) ++seg;
                const uint32_t tO = tmem + (seg & 1) * 2 * NP;
                if (!mbar_wait(&ctrl->p_full[i & 1], (i >> 1) & 1, &ctrl->abort)) {
                    fail(p, ctrl, kErrWaitTimeout, kSitePFull, i);
                    report(p, kRolePV, kSitePFull, i);
                    break;
                }
                tc_fence_after();
                if (mt == 0) MLA_TRACE_POINT(i, kTrPvIssue);
                const uint64_t dp = smem_desc(smem_u32(pbufs + (i % C::kPBufs) * C::kPBytes), C::kPBlockBytes, p_sbo,
                                              C::kPSwizzle);
                const int slot = (2 * i + mt) % C::kRL;
                const uint64_t da = smem_desc(smem_u32(pair_ring + slot * C::kPairBytes), 16384, 1024, kSw128);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    umma_bf16(tO + mt * NP, da + ((kk * 2048) >> 4), dp + ((kk * 16 * C::kNH * 2) >> 4), idPV,
                              (new_seg && kk == 0) ? 0u : 1u);
                umma_commit(&ctrl->pair_empty[slot]);
                umma_commit(&ctrl->o_done[i & 1]);
                if (p.test_hold == 2 && mt == 1 && i < 32) spin_for_ns(20000);  // test hook: a lagging issuer
                if (mt == 0) MLA_TRACE_POINT(i, kTrPvIssued);
                it.next(p.seq_lens, p.B);
            }
        } else if (!LSU && warp == 1) {
            // ------------------------------------------------- TMA producer
            // Lane r owns run r of the tile (a page-contiguous run of BR rows).
            TileIt it;
            it.init(p.seq_lens, ctrl->b0, ctrl->j0);
            const uint64_t pol = l2_policy_evict_first();
            const int BR = p.run_rows;
            bool bad = false, ok = true;
            int fsite = 0, ftile = 0;
            for (int i = 0; i < ntiles && ok; ++i) {
                const int valid = min(kTile, it.T - it.j * kTile);
                const int nruns = (valid + BR - 1) / BR;
                const int32_t* btr = p.block_table + static_cast<int64_t>(it.b) * p.bt_stride;
                const int y = lane < nruns ? static_cast<int>(token_slot(p, btr, it.j * kTile + lane * BR, bad)) : 0;
                const uint32_t chunk_bytes = static_cast<uint32_t>(nruns * BR * 128);
                if (lane == 0) MLA_TRACE_POINT(i, kTrProdStart);
                for (int pp = 0; pp < 2; ++pp) {
                    const int u = 2 * i + pp, slot = u % C::kRL;
                    if (u >= C::kRL &&
                        !__all_sync(0xffffffffu, mbar_wait(&ctrl->pair_empty[slot], ((u / C::kRL) - 1) & 1, &ctrl->abort))) {
                        ok = false;
                        fsite = kSiteTmaPairEmpty;
                        ftile = i;
                        break;
                    }
                    if constexpr (KIND == 0) {
                        if (lane == 0) mbar_arrive_expect_tx(&ctrl->pair_full[slot], 2 * chunk_bytes);
                        __syncwarp();
                        if (lane < nruns) {
                            uint8_t* dst = pair_ring + slot * C::kPairBytes + lane * BR * 128;
#pragma unroll
                            for (int c = 0; c < 2; ++c)
                                tma_load_2d(dst + c * 16384, &tmap_lat, &ctrl->pair_full[slot],
                                            256 * rank + 128 * pp + 64 * c, y, pol);
                        }
                    }
                }
                if (!ok) break;
                if constexpr (KIND == 1) {
                    // this CTA's 256 codes of each row ([row][256 B]) into the first
                    // pair slot, the row's four scales ([row][16 B]) into the second
                    const int s0 = (2 * i) % C::kRL, s1 = (2 * i + 1) % C::kRL;
                    uint64_t* rb = &ctrl->raw_full[i % kRawSlots];
                    if (lane == 0) mbar_arrive_expect_tx(rb, static_cast<uint32_t>(nruns * BR * (256 + 16)));
                    __syncwarp();
                    if (lane < nruns) {
                        tma_load_2d(pair_ring + s0 * C::kPairBytes + lane * BR * 256, &tmap_lat, rb, 256 * rank, y, pol);
                        tma_load_2d(pair_ring + s1 * C::kPairBytes + lane * BR * 16, &maps.aux, rb, 512, y, pol);
                    }
                }
                if (!ok) break;
                const int rr = i % C::kRR;
                if (i >= C::kRR &&
                    !__all_sync(0xffffffffu, mbar_wait(&ctrl->rope_empty[rr], ((i / C::kRR) - 1) & 1, &ctrl->abort))) {
                    ok = false;
                    fsite = kSiteTmaRopeEmpty;
                    ftile = i;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(&ctrl->rope_full[rr], chunk_bytes / 2);
                __syncwarp();
                if (lane < nruns)
                    tma_load_2d(rope_ring + rr * C::kRopeBytes + lane * BR * 64, &tmap_rope, &ctrl->rope_full[rr],
                                (KIND == 0 ? 512 : 264) + 32 * rank, y, pol);
                if (lane == 0) MLA_TRACE_POINT(i, kTrProdIssued);
                it.next(p.seq_lens, p.B);
            }
            if (!ok && lane == 0) {
                fail(p, ctrl, kErrWaitTimeout, fsite, ftile);
                report(p, kRoleTma, fsite, ftile);
            }
            if (bad) atomicOr(status_rec(p), kErrBadBlock);
        } else if (!LSU && KIND == 1 && warp >= 8) {
            // ------------------------------------------------- fp8 expand warps
            // Warp 8 + w expands rows [32w, 32w + 32) of each tile: two rows per
            // step, a lane per 16 codes. All rows are read into registers and
            // the four warps meet before any bf16 is written over the codes.
            const int cw = warp - 8;
            bool ok = true;
            int ftile = 0;
            for (int i = 0; i < ntiles; ++i) {
                const int s0 = (2 * i) % C::kRL, s1 = (2 * i + 1) % C::kRL;
                if (!__all_sync(0xffffffffu,
                                mbar_wait(&ctrl->raw_full[i % kRawSlots], (i / kRawSlots) & 1, &ctrl->abort))) {
                    ok = false;
                    ftile = i;
                }
                // every expand warp reaches the barriers below, so a timeout in
                // one warp cannot strand the others
                if (!named_bar_and(4, 128, ok ? 1 : 0)) {
                    ok = false;
                    break;
                }
                const uint8_t* codes = pair_ring + s0 * C::kPairBytes;
                const uint8_t* scales = pair_ring + s1 * C::kPairBytes;
                const int unit = lane & 15;
                uint4 v[16];
                float sc[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int row = 32 * cw + 2 * k + (lane >> 4);
                    v[k] = *reinterpret_cast<const uint4*>(codes + row * 256 + unit * 16);
                    sc[k] = *reinterpret_cast<const float*>(scales + row * 16 + 4 * (2 * rank + (unit >> 3)));
                }
                named_bar_sync(4, 128);
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int row = 32 * cw + 2 * k + (lane >> 4);
                    uint4 lo, hi;
                    dequant16(v[k], sc[k], lo, hi);
                    // dims 16*unit .. +16 of this CTA's 256: chunk unit/4 (64 dims),
                    // 16-byte units 2*(unit%4), +1 within the 128-byte row
                    const int c = unit >> 2, un = (unit & 3) * 2;
                    uint8_t* rowp = pair_ring + (c < 2 ? s0 : s1) * C::kPairBytes + (c & 1) * 16384 + row * 128;
                    *reinterpret_cast<uint4*>(rowp + ((un ^ (row & 7)) << 4)) = lo;
                    *reinterpret_cast<uint4*>(rowp + (((un + 1) ^ (row & 7)) << 4)) = hi;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&ctrl->pair_full[s0]);
                    mbar_arrive(&ctrl->pair_full[s1]);
                }
            }
            if (!ok && lane == 0) {
                fail(p, ctrl, kErrWaitTimeout, kSiteRawFull, ftile);
                report(p, kRoleLsu0 + cw, kSiteRawFull, ftile);
            }
        } else if (LSU && warp >= 8) {
            // ------------------------------------- load/convert producers
            // Each warp keeps a fixed, in-order share of every tile: warps 8/9 the
            // two 64-row halves of pair 0, warps 10/11 those of pair 1, and each a
            // 32-row quarter of the rope half. Walking the tiles in order, a warp
            // never waits on a slot more than one phase ahead of its release.
            // Rows past the request are left stale (the softmax clears them).
            const int pw = warp - 8;
            const int pk = pw >> 1, half = pw & 1;
            TileIt it;
            it.init(p.seq_lens, ctrl->b0, ctrl->j0);
            TileIt pf = it;
            int pf_i = 0;
            bool bad = false, ok = true;
            const int rb = KIND == 0 ? kRowBf16 : kRowFp8;
            int fsite = 0, ftile = 0;
            if (pw == 0 && lane == 0) prefetch_tile(p, pf, rb, rank);
            for (int i = 0; i < ntiles && ok; ++i) {
                if (pw == 0 && lane == 0) {
                    while (pf_i < i + kPrefetchTiles && pf_i + 1 < ntiles) {
                        pf.next(p.seq_lens, p.B);
                        ++pf_i;
                        prefetch_tile(p, pf, rb, rank);
                    }
                }
                const int valid = min(kTile, it.T - it.j * kTile);
                const int32_t* btr = p.block_table + static_cast<int64_t>(it.b) * p.bt_stride;
                // ---- pair pk, rows [64*half, 64*half + 64)
                {
                    const int u = 2 * i + pk, slot = u % C::kRL;
                    if (u >= C::kRL &&
                        !__all_sync(0xffffffffu, mbar_wait(&ctrl->pair_empty[slot], ((u / C::kRL) - 1) & 1, &ctrl->abort))) {
                        ok = false;
                        fsite = kSiteLsuPairEmpty;
                        ftile = i;
                        break;
                    }
                    uint8_t* dst = pair_ring + slot * C::kPairBytes;
                    const int r0 = 64 * half, r1 = min(64 * half + 64, valid);
                    if (KIND == 0) {
                        // 16 units of 16 B per token: dims 256*rank + 128*pk + [0, 128)
                        for (int q0 = r0 * 16; q0 < r1 * 16; q0 += 256) {
                            uint4 v[8];
                            int tl[8], uu[8];
#pragma unroll
                            for (int s8 = 0; s8 < 8; ++s8) {
                                const int q = q0 + s8 * 32 + lane;
                                tl[s8] = q >> 4;
                                uu[s8] = q & 15;
                                if (tl[s8] < r1) {
                                    const int64_t slot64 = token_slot(p, btr, it.j * kTile + tl[s8], bad);
                                    v[s8] = __ldg(reinterpret_cast<const uint4*>(p.cache + slot64 * rb + 512 * rank + pk * 256) + uu[s8]);
                                }
                            }
#pragma unroll
                            for (int s8 = 0; s8 < 8; ++s8)
                                if (tl[s8] < r1) {
                                    const int c = uu[s8] >> 3, un = uu[s8] & 7;
                                    *reinterpret_cast<uint4*>(dst + c * 16384 + tl[s8] * 128 + ((un ^ (tl[s8] & 7)) << 4)) = v[s8];
                                }
                        }
                    } else {
                        // quant block 2*rank + pk: 8 units of 16 codes per token and its scale
                        const int qb = 2 * rank + pk;
                        for (int q0 = r0 * 8; q0 < r1 * 8; q0 += 256) {
                            uint4 v[8];
                            float sc[8];
                            int tl[8], uu[8];
#pragma unroll
                            for (int s8 = 0; s8 < 8; ++s8) {
                                const int q = q0 + s8 * 32 + lane;
                                tl[s8] = q >> 3;
                                uu[s8] = q & 7;
                                if (tl[s8] < r1) {
                                    const int64_t slot64 = token_slot(p, btr, it.j * kTile + tl[s8], bad);
                                    const uint8_t* row = p.cache + slot64 * rb;
                                    v[s8] = __ldg(reinterpret_cast<const uint4*>(row + qb * 128) + uu[s8]);
                                    sc[s8] = __ldg(reinterpret_cast<const float*>(row + 512) + qb);
                                }
                            }
#pragma unroll
                            for (int s8 = 0; s8 < 8; ++s8)
                                if (tl[s8] < r1) {
                                    uint4 lo, hi;
                                    dequant16(v[s8], sc[s8], lo, hi);
                                    const int c = uu[s8] >> 2, un = (uu[s8] & 3) * 2;
                                    uint8_t* rowp = dst + c * 16384 + tl[s8] * 128;
                                    *reinterpret_cast<uint4*>(rowp + ((un ^ (tl[s8] & 7)) << 4)) = lo;
                                    *reinterpret_cast<uint4*>(rowp + (((un + 1) ^ (tl[s8] & 7)) << 4)) = hi;
                                }
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctrl->pair_full[slot]);
                }
                // ---- rope half, rows [32*pw, 32*pw + 32)
                {
                    const int rr = i % C::kRR;
                    if (i >= C::kRR &&
                        !__all_sync(0xffffffffu, mbar_wait(&ctrl->rope_empty[rr], ((i / C::kRR) - 1) & 1, &ctrl->abort))) {
                        ok = false;
                        fsite = kSiteLsuRopeEmpty;
                        ftile = i;
                        break;
                    }
                    uint8_t* dst = rope_ring + rr * C::kRopeBytes;
                    const int roff = (KIND == 0 ? 1024 : 528) + 64 * rank;
                    const int r0 = 32 * pw, r1 = min(32 * pw + 32, valid);
                    for (int q0 = r0 * 4; q0 < r1 * 4; q0 += 128) {
                        uint4 v[4];
                        int tl[4], uu[4];
#pragma unroll
                        for (int s4 = 0; s4 < 4; ++s4) {
                            const int q = q0 + s4 * 32 + lane;
                            tl[s4] = q >> 2;
                            uu[s4] = q & 3;
                            if (tl[s4] < r1) {
                                const int64_t slot64 = token_slot(p, btr, it.j * kTile + tl[s4], bad);
                                v[s4] = __ldg(reinterpret_cast<const uint4*>(p.cache + slot64 * rb + roff) + uu[s4]);
                            }
                        }
#pragma unroll
                        for (int s4 = 0; s4 < 4; ++s4)
                            if (tl[s4] < r1)
                                *reinterpret_cast<uint4*>(dst + tl[s4] * 64 + ((uu[s4] ^ ((tl[s4] >> 1) & 3)) << 4)) = v[s4];
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctrl->rope_full[rr]);
                }
                it.next(p.seq_lens, p.B);
            }
            if (!ok && lane == 0) {
                fail(p, ctrl, kErrWaitTimeout, fsite, ftile);
                report(p, kRoleLsu0 + pw, fsite, ftile);
            }
            if (bad) atomicOr(status_rec(p), kErrBadBlock);
        } else if (warp >= 4 && warp < 8) {
            // ------------------------------------------ softmax + epilogue
            const int st = threadIdx.x - 128;  // token row of the tile / TMEM lane
            const int sw = warp - 4;
            const uint32_t lane_base = static_cast<uint32_t>(sw * 32) << 16;
            const int peer = rank ^ 1;
            const uint32_t x_local = smem_u32(xbuf);
            const uint32_t x_peer = mapa_shared(x_local, peer);
            const uint32_t xfull_peer = mapa_shared(smem_u32(&ctrl->xfull), peer);
            const uint32_t xfree_peer = mapa_shared(smem_u32(&ctrl->xfree), peer);
            // Softmax columns of this CTA: [own0, own0 + NH); the partial scores of
            // [snd0, snd0 + NH) go to the peer (all columns when not split).
            constexpr int NH = C::kNH;
            constexpr uint32_t kXferBytes = 128 * NH * 4;
            const int own0 = C::kSplit ? rank * NH : 0;
            const int snd0 = C::kSplit ? peer * NH : 0;
            // 16-byte unit swizzle of the exchange rows (NH/4 units per row)
            const int xs = (NH == 16) ? ((st >> 1) & 3) : (st & 7);
            TileIt it;
            it.init(p.seq_lens, ctrl->b0, ctrl->j0);
            float l[NH];
#pragma unroll
            for (int c = 0; c < NH; ++c) l[c] = 0.f;
            int seg_start_j = it.j;
            bool seg_has_pv = false;
            int seg = 0;               // segment index: its O accumulator is (seg & 1)
            uint32_t obuf = 0;         // column of the current O accumulator
            // The segment that ended with the previous tile: its row sums and maxima
            // are captured, its output is written out once its last PV is done.
            bool pend = false;
            bool pend_final = false;
            int pend_b = 0;
            // Output rows being drained from an O accumulator a few columns per
            // tile: plain stores that the memory pipe absorbs in the background
            // (a whole segment at once would stall the group behind the cache stream).
            int dr_left = 0, dr_step = 0, dr_b = 0;
            bool dr_final = false;
            uint32_t dr_obuf = 0;
            constexpr int kDC = 8;  // columns per drain step
            // rows (in this row group) of the segment being drained, and the drain
            // steps per 128-dim half: recomputed from dr_b where needed, so
            // nothing more stays live across the tile loop
            auto dr_rows = [&]() { return req_rows_in_group(p, dr_b, gy); };

            // O columns [col0, col0 + NH) of accumulator ob, both 128-dim halves,
            // times alpha[0 .. NH) (the caller has waited for the last PV into it)
            auto rescale_o = [&](uint32_t ob, int col0, const float* alpha) {
                tc_fence_after();
                __syncwarp();
#pragma unroll 1
                for (int mt = 0; mt < 2; ++mt)
#pragma unroll 1
                    for (int c0 = 0; c0 < NH; c0 += 16) {
                        uint32_t o[16];
                        tmem_ld_x16(tmem + lane_base + ob + mt * NP + col0 + c0, o);
#pragma unroll
                        for (int cc = 0; cc < 16; ++cc) o[cc] = __float_as_uint(__uint_as_float(o[cc]) * alpha[c0 + cc]);
                        tmem_st_x16(tmem + lane_base + ob + mt * NP + col0 + c0, o);
                    }
                tmem_wait_st();
            };

            // This CTA's half of the NP query rows of request bq (row group gy)
            // by TMA, in the layout S reads as its B operand: latent chunks
            // 256*rank + 64k (k = 0..3) K-major with 128-B swizzle at k*NP*128,
            // then the rope half (32 dims) with 64-B swizzle at 4*NP*128. Rows
            // past the group's real rows belong to other requests (or are zero
            // past the end); their score columns are masked to -inf.
            auto issue_q = [&](int bq) {
                const int y = static_cast<int>(req_row0(p, bq) + gy * 64);
                const uint64_t pol = l2_policy_evict_first();
                mbar_arrive_expect_tx(&ctrl->q_full, C::kQBytes);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    tma_load_2d(qs + k * NP * 128, &maps.q, &ctrl->q_full, 256 * rank + 64 * k, y, pol);
                tma_load_2d(qs + 4 * NP * 128, &maps.qpe, &ctrl->q_full, 32 * rank, y, pol);
            };

            // Row sums and maxima of segment sg, which just ended, into
            // dlt[sg & 1] / dm (this CTA's columns; with split columns the sums
            // also go to the peer, whose drain needs every column's), then fresh
            // softmax state for the next segment.
            auto capture = [&](int i, int sg) {
                if (st == 0) MLA_TRACE_POINT(i, kTrEpiStart);
#pragma unroll
                for (int c = 0; c < NH; ++c) {
                    const float v = warp_sum(l[c]);
                    if (lane == 0) ctrl->red[sw][c] = v;
                }
                named_bar_sync(1, 128);
                float* dl = ctrl->dlt[sg & 1];
                if (st < NH) {
                    const int c = own0 + st;
                    dl[c] = ctrl->red[0][st] + ctrl->red[1][st] + ctrl->red[2][st] + ctrl->red[3][st];
                    ctrl->dm[c] = ctrl->m[c];
                    ctrl->m[c] = -INFINITY;
                }
#pragma unroll
                for (int c = 0; c < NH; ++c) l[c] = 0.f;
                named_bar_sync(1, 128);
                if constexpr (C::kSplit) {
                    if (st == 0) mbar_arrive_expect_tx(&ctrl->dfull[sg & 1], NH * 4);
                    if (st < NH / 4) {
                        const float4 v = reinterpret_cast<const float4*>(dl + own0)[st];
                        st_async_v4(mapa_shared(smem_u32(dl + own0 + 4 * st), peer), __float_as_uint(v.x),
                                    __float_as_uint(v.y), __float_as_uint(v.z), __float_as_uint(v.w),
                                    mapa_shared(smem_u32(&ctrl->dfull[sg & 1]), peer));
                    }
                }
                if (st == 0) MLA_TRACE_POINT(i, kTrEpiRed);
            };

            // The captured segment sg (accumulator src) has finished its last
            // PV: write the LSE of this CTA's columns and start draining its rows
            // (every column, once the peer's row sums are in).
            int dr_sg = 0;
            auto start_drain = [&](uint32_t src, int sg, int i, int sb, bool sfinal) {
                if constexpr (C::kSplit) group_wait(&ctrl->dfull[sg & 1], (sg >> 1) & 1, p, ctrl, kSiteDFull, i, true);
                const int64_t pslot = static_cast<int64_t>(gy) * p.SPG + g + sb;
                const int shq = req_rows_in_group(p, sb, gy);
                const int c = own0 + st;
                if (st < NH && c < shq && (C::kSplit || rank == 0)) {
                    const float lt = ctrl->dlt[sg & 1][c];
                    const float lv = lt > 0.f ? (ctrl->dm[c] + log2f(lt)) * kLn2 : -INFINITY;
                    if (sfinal) p.lse[req_row0(p, sb) + gy * 64 + c] = lv;
                    else p.part_lse[pslot * 64 + c] = lv;
                }
                dr_left = 2 * ((shq + kDC - 1) / kDC);
                dr_step = 0;
                dr_b = sb;
                dr_final = sfinal;
                dr_obuf = src;
                dr_sg = sg;
                pend = false;
            };

            // One drain step: kDC columns of one 128-dim half, O / l, into the
            // output rows (a whole request) or the cluster's partial slot.
            auto drain_step = [&]() {
                const int dr_hq = dr_rows();
                const int dr_per_half = (dr_hq + kDC - 1) / kDC;
                const int mt = dr_step / dr_per_half;
                const int c0 = (dr_step - mt * dr_per_half) * kDC;
                uint32_t o[kDC];
                tmem_ld_x8(tmem + lane_base + dr_obuf + mt * NP + c0, o);
                // lane st holds dim 256 rank + 128 mt + st; each quad of lanes
                // transposes 4 x 4 blocks so that a lane stores 4 consecutive dims
                // of one row in one 16-byte store
                const int64_t dq = 256 * rank + 128 * mt + (st & ~3);
                const int64_t pslot = static_cast<int64_t>(gy) * p.SPG + g + dr_b;
#pragma unroll
                for (int cb = 0; cb < kDC; cb += 4) {
                    float x[4] = {__uint_as_float(o[cb]), __uint_as_float(o[cb + 1]), __uint_as_float(o[cb + 2]),
                                  __uint_as_float(o[cb + 3])};
                    quad_transpose(x, lane);
                    const int c = c0 + cb + (lane & 3);
                    if (c < dr_hq) {
                        const float lt = ctrl->dlt[dr_sg & 1][c];
                        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (lt > 0.f) v = make_float4(x[0] / lt, x[1] / lt, x[2] / lt, x[3] / lt);
                        if (dr_final) {
                            const int64_t idx = (req_row0(p, dr_b) + gy * 64 + c) * kD + dq;
                            if (p.out_f32)
                                *reinterpret_cast<float4*>(static_cast<float*>(p.out) + idx) = v;
                            else
                                *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + idx) =
                                    make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
                        } else {
                            *reinterpret_cast<float4*>(p.part_o + (pslot * 64 + c) * kD + dq) = v;
                        }
                    }
                }
                ++dr_step;
                --dr_left;
            };

            // The request and kind of the segment captured last (drained once its
            // last PV is done).
            int cap_b = 0;
            bool cap_final = false;

            // Hand tile t to the PV issuer: with split columns, wait for the peer's
            // P block and message and apply its rescale to this CTA's O first;
            // then start or advance the drain. False when the group aborts.
            auto finish = [&](int t) -> bool {
                if constexpr (C::kSplit) {
                    const int fpb = t % C::kPBufs;
                    group_wait(&ctrl->pin[fpb], (t / C::kPBufs) & 1, p, ctrl, kSitePIn, t, true);
                    if (ctrl->pflag[fpb][0] && seg_has_pv) {
                        group_wait(&ctrl->o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, p, ctrl, kSiteORescale, t);
                        rescale_o(obuf, snd0, ctrl->palpha[fpb]);
                        tc_fence_before();
                    }
                    named_bar_sync(1, 128);
                }
                if (ctrl->abort) return false;  // same value in every thread after the barrier
                if (st == 0) {
                    MLA_TRACE_POINT(t, kTrSmPArrive);
                    MLA_TTRACE(t);
                    // the test hook withholds tile 0, so the PV issuers' bounded wait
                    // gives up and every role leaves through the abort path
                    if (!(p.test_hold == 1 && t == 0)) mbar_arrive(&ctrl->p_full[t & 1]);
                }
                seg_has_pv = true;
                if (pend) {
                    // PV(t-1), the captured segment's last, is long done by now
                    group_wait(&ctrl->o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, p, ctrl, kSiteOEpi, t);
                    tc_fence_after();
                    start_drain(obuf ^ (2 * NP), seg - 1, t, cap_b, cap_final);
                    if (st == 0) MLA_TRACE_POINT(t, kTrEpiStored);
                } else if (dr_left > 0) {
                    tc_fence_after();
                    drain_step();
                    tc_fence_before();
                }
                return true;
            };

            if (st == 0) issue_q(it.b);
            bool alive = true;
            for (int i = 0; i < ntiles; ++i) {
                const int b = it.b, j = it.j, T = it.T;
                const bool last_of_seg = (j == it.tiles - 1) || (i == ntiles - 1);
                group_wait(&ctrl->s_full[i & 1], (i >> 1) & 1, p, ctrl, kSiteSFull, i);
                if (st == 0) {
                    MLA_TRACE_POINT(i, kTrSmSFull);
                    if (last_of_seg && i + 1 < ntiles) {
                        // S(i) is complete, so Q may be replaced by the next request's
                        TileIt nx = it;
                        nx.next(p.seq_lens, p.B);
                        issue_q(nx.b);
                    }
                }
                tc_fence_after();
                __syncwarp();
                uint32_t sr[NP];
                tmem_ld_np<NP>(tmem + lane_base + C::kColS + (i & 1) * NP, sr);
                tc_fence_before();
                // partial score of own column k / of the peer's column k (indices
                // stay compile-time constants so sr[] remains in registers)
                auto own_s = [&](int k) -> uint32_t {
                    if constexpr (C::kSplit) return rank ? sr[NH + k] : sr[k];
                    else return sr[k];
                };
                auto snd_s = [&](int k) -> uint32_t {
                    if constexpr (C::kSplit) return rank ? sr[k] : sr[NH + k];
                    else return sr[k];
                };
                if (st == 0) MLA_TRACE_POINT(i, kTrSmTmemLd);
                if (st == 0 && (i == 0 || j == 0) && !last_of_seg) {
                    // warm L2 with the next request's queries and page list
                    TileIt nx = it;
                    nx.j = nx.tiles - 1;
                    nx.next(p.seq_lens, p.B);
                    if (nx.b < p.B) prefetch_request(p, nx.b, gy);
                }
                // send this CTA's partial scores once the peer has read the last ones
                if (i > 0) group_wait(&ctrl->xfree, (i - 1) & 1, p, ctrl, kSiteXFree, i, true);
                if constexpr (C::kSendInP) {
                    // the staging goes into this tile's P buffer: PV(i - kPBufs) has read it
                    if (i >= C::kPBufs)
                        group_wait(&ctrl->o_done[(i - C::kPBufs) & 1], ((i - C::kPBufs) >> 1) & 1, p, ctrl, kSiteOPbuf, i);
                }
                if (st == 0) MLA_TRACE_POINT(i, kTrSmXFree);
                {
                    // stage columns [snd0, snd0 + NH) of the row in the send buffer
                    // (the peer's exchange-buffer layout); one thread pushes the block
                    uint8_t* sendb = C::kSendInP ? pbufs + (i % C::kPBufs) * C::kPBytes : smem + C::kOffSend;
#pragma unroll
                    for (int u = 0; u < NH / 4; ++u)
                        *reinterpret_cast<uint4*>(sendb + st * NH * 4 + ((u ^ xs) << 4)) =
                            make_uint4(snd_s(4 * u), snd_s(4 * u + 1), snd_s(4 * u + 2), snd_s(4 * u + 3));
                    fence_proxy_async_smem();
                    named_bar_sync(1, 128);
                    if (st == 0) {
                        mbar_arrive_expect_tx(&ctrl->xfull, kXferBytes);
                        bulk_s2cluster(x_peer, sendb, kXferBytes, xfull_peer);
                    }
                }
                if (st == 0) MLA_TRACE_POINT(i, kTrSmSent);
                if (i > 0 && j == 0) {
                    // the previous segment ended with tile i-1. The older one still
                    // draining (if any) finishes first: its accumulator is the one
                    // this segment will use, and dlt / dm are about to be replaced.
                    if (dr_left > 0) {
                        tc_fence_after();
                        while (dr_left > 0) drain_step();
                        tc_fence_before();
                    }
                    if (st == 0) MLA_TRACE_POINT(i, kTrEpiHalf);
                    capture(i, seg);
                    pend = true;
                    cap_b = pend_b;
                    cap_final = pend_final;
                    seg_has_pv = false;
                    ++seg;
                    obuf = (seg & 1) * 2 * NP;
                }
                group_wait(&ctrl->xfull, i & 1, p, ctrl, kSiteXFull, i, true);
                if (st == 0) MLA_TRACE_POINT(i, kTrSmXFull);
                // x[k]: full score of column own0 + k
                float x[NH];
#pragma unroll
                for (int u = 0; u < NH / 4; ++u) {
                    const float4 v = *reinterpret_cast<const float4*>(xbuf + st * NH * 4 + ((u ^ xs) << 4));
                    x[4 * u] = __uint_as_float(own_s(4 * u)) + v.x;
                    x[4 * u + 1] = __uint_as_float(own_s(4 * u + 1)) + v.y;
                    x[4 * u + 2] = __uint_as_float(own_s(4 * u + 2)) + v.z;
                    x[4 * u + 3] = __uint_as_float(own_s(4 * u + 3)) + v.w;
                }
                if (st == 0) MLA_TRACE_POINT(i, kTrSmXRead);

                const int tok = j * kTile + st;
                // this tile's request: its verify length and its rows in this row group
                const int seg_qt = req_qt(p, b), seg_hq = req_rows_in_group(p, b, gy);
                const bool all_vis = (j * kTile + kTile + seg_qt - 1) <= T;
                const float4* m4 = reinterpret_cast<const float4*>(ctrl->m + own0);
                if (all_vis) {
                    // every real row sees every token of the tile
#pragma unroll
                    for (int c = 0; c < NH; ++c) x[c] = (own0 + c < seg_hq) ? x[c] * p.scale_log2 : -INFINITY;
                } else {
                    // tail of a request: query token r / Hq of the step sees tokens up to
                    // T - Qt + r / Hq, and rows past the request's are padding
                    if (p.cu_q) {
#pragma unroll
                        for (int c = 0; c < NH; ++c) {
                            const int r = gy * 64 + own0 + c;
                            const bool v = own0 + c < seg_hq && tok + seg_qt - 1 - r / p.Hq < T;
                            x[c] = v ? x[c] * p.scale_log2 : -INFINITY;
                        }
                    } else {
                        // the same limits, tabulated once (every request has p.Qt tokens)
#pragma unroll
                        for (int c = 0; c < NH; ++c)
                            x[c] = (tok + ctrl->colvis[own0 + c] < T) ? x[c] * p.scale_log2 : -INFINITY;
                    }
                }
                int need = 0;
#pragma unroll
                for (int u = 0; u < NH / 4; ++u) {
                    const float4 mv = m4[u];
                    need |= (x[4 * u] > mv.x + kRescaleThreshold) | (x[4 * u + 1] > mv.y + kRescaleThreshold) |
                            (x[4 * u + 2] > mv.z + kRescaleThreshold) | (x[4 * u + 3] > mv.w + kRescaleThreshold);
                }
                // (also: every thread has read the exchange buffer; hand it back to the peer)
                if (st == 0) MLA_TRACE_POINT(i, kTrSmMath);
                need = named_bar_or(2, 128, need);
                if (st == 0) {
                    MLA_TRACE_POINT(i, kTrSmBarOr);
                    // every thread has read S(i) from TMEM (fenced before the barrier)
                    // and has used the peer's scores read from the exchange buffer
                    mbar_arrive(&ctrl->s_free[i & 1]);
                    mbar_arrive_remote_relaxed(xfree_peer);
                }
                if (need) {
#pragma unroll
                    for (int c = 0; c < NH; ++c) {
                        const float v = warp_max(x[c]);
                        if (lane == 0) ctrl->red[sw][c] = v;
                    }
                    named_bar_sync(1, 128);
                    if (st < NH) {
                        const int c = own0 + st;
                        const float mt = fmaxf(fmaxf(ctrl->red[0][st], ctrl->red[1][st]),
                                               fmaxf(ctrl->red[2][st], ctrl->red[3][st]));
                        const float mo = ctrl->m[c];
                        const float mn = fmaxf(mo, mt);
                        ctrl->alpha[c] = (mo == -INFINITY) ? 0.f : ex2(mo - mn);
                        ctrl->m[c] = mn;
                    }
                    named_bar_sync(1, 128);
#pragma unroll
                    for (int c = 0; c < NH; ++c) l[c] *= ctrl->alpha[own0 + c];
                    if (seg_has_pv) {
                        // O holds earlier tiles of this segment: wait for their PV, rescale
                        group_wait(&ctrl->o_done[(i - 1) & 1], ((i - 1) >> 1) & 1, p, ctrl, kSiteORescale, i);
                        rescale_o(obuf, own0, ctrl->alpha + own0);
                    }
                }
#pragma unroll
                for (int u = 0; u < NH / 4; ++u) {
                    const float4 mv = m4[u];
                    const float mm[4] = {mv.x, mv.y, mv.z, mv.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        // masked entries are -inf: ex2(-inf - finite) = 0 exactly; a row
                        // with no visible token yet has m = -inf, replaced by 0 here
                        const int c = 4 * u + k;
                        const float mk = (mm[k] == -INFINITY) ? 0.f : mm[k];
                        const float pc = ex2(x[c] - mk);
                        l[c] += pc;
                        x[c] = pc;
                    }
                }
                if (st == 0) MLA_TRACE_POINT(i, kTrSmExpLoop);
                // The P buffer of this tile was last read by PV(i - kPBufs). Each warp
                // writes its own 32 rows, so one lane per warp waits; on a timeout the
                // warp carries on to the next group barrier, which then fails for all.
                if (i >= C::kPBufs) {
                    const int jp = i - C::kPBufs;
                    bool okp = true;
                    if (lane == 0) okp = !ctrl->abort && mbar_wait(&ctrl->o_done[jp & 1], (jp >> 1) & 1, &ctrl->abort);
                    okp = __shfl_sync(0xffffffffu, okp ? 1 : 0, 0) != 0;
                    if (!okp && lane == 0) fail(p, ctrl, kErrWaitTimeout, kSiteOPbuf, i);
                }
                if constexpr (C::kSendInP) {
                    // the peer has consumed this tile's scores, so the bulk copy has
                    // read the staging that P is about to replace
                    group_wait(&ctrl->xfree, i & 1, p, ctrl, kSiteXFree, i, true);
                }
                if (st == 0) MLA_TRACE_POINT(i, kTrSmExp);
                const int pb = i % C::kPBufs;
                if constexpr (C::kSplit) {
                    // this CTA's PV(i - kPBufs) is done: the peer may write its P
                    // block of tile i into this CTA's P buffer
                    if (st == 0 && i >= C::kPBufs)
                        mbar_arrive_remote_relaxed(mapa_shared(smem_u32(&ctrl->rp_free[pb]), peer));
                    if (st == 0) mbar_arrive_expect_tx(&ctrl->pin[pb], C::kPBlockBytes + NH * 4 + 16);
                }
                // P row `st` of this CTA's column block: NH bf16, MN-major, swizzled
                // as the MMA reads it
                uint8_t* pblk = pbufs + pb * C::kPBytes + (own0 / NH) * C::kPBlockBytes;
                uint8_t* prow = pblk + st * NH * 2;
                const int sz = swz_p(st, C::kPSwizzle);
#pragma unroll
                for (int u = 0; u < NH / 8; ++u) {
                    const uint4 v = make_uint4(pack_bf16x2(x[8 * u + 0], x[8 * u + 1]), pack_bf16x2(x[8 * u + 2], x[8 * u + 3]),
                                               pack_bf16x2(x[8 * u + 4], x[8 * u + 5]), pack_bf16x2(x[8 * u + 6], x[8 * u + 7]));
                    *reinterpret_cast<uint4*>(prow + ((u ^ sz) << 4)) = v;
                }
                if (j * kTile + kTile > T) {
                    // rows past the request hold stale data (maybe NaN); P is 0 there,
                    // but 0 * NaN would still poison O, so clear them. In each 64-dim
                    // chunk the token rows r0..127 are one contiguous range; the 128
                    // threads write consecutive 16-byte units of it.
                    const int r0 = max(T - j * kTile, 0);
                    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                    const int nunits = (kTile - r0) * 8;  // 16-byte units per chunk
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint8_t* base = pair_ring + ((2 * i + (q >> 1)) % C::kRL) * C::kPairBytes + (q & 1) * 16384 + r0 * 128;
                        for (int u = st; u < nunits; u += 128) *reinterpret_cast<uint4*>(base + u * 16) = z;
                    }
                }
                if (st == 0) MLA_TRACE_POINT(i, kTrSmPStore);
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar_sync(1, 128);
                if constexpr (C::kSplit) {
                    if (st == 0 && !ctrl->abort) {
                        // push this CTA's P block and rescale message into the peer's
                        // P buffer once its PV(i - kPBufs) is done
                        bool okr = true;
                        if (i >= C::kPBufs)
                            okr = mbar_wait_cluster(&ctrl->rp_free[pb], ((i / C::kPBufs) - 1) & 1, &ctrl->abort);
                        if (!okr) {
                            fail(p, ctrl, kErrWaitTimeout, kSiteRpFree, i);
                            report(p, kRoleSoftmax, kSiteRpFree, i);
                        } else {
                            const uint32_t pin_peer = mapa_shared(smem_u32(&ctrl->pin[pb]), peer);
                            bulk_s2cluster(mapa_shared(smem_u32(pblk), peer), pblk, C::kPBlockBytes, pin_peer);
                            const uint32_t* al = reinterpret_cast<const uint32_t*>(ctrl->alpha + own0);
                            const uint32_t pa = mapa_shared(smem_u32(ctrl->palpha[pb]), peer);
#pragma unroll
                            for (int u = 0; u < NH / 4; ++u)
                                st_async_v4(pa + 16 * u, al[4 * u], al[4 * u + 1], al[4 * u + 2], al[4 * u + 3], pin_peer);
                            st_async_v4(mapa_shared(smem_u32(ctrl->pflag[pb]), peer), static_cast<uint32_t>(need), 0u,
                                        0u, 0u, pin_peer);
                        }
                    }
                }
                if (!finish(i)) {
                    alive = false;
                    break;
                }
                if (last_of_seg) {
                    pend_final = (seg_start_j == 0) && (j == it.tiles - 1);
                    pend_b = b;
                    seg_start_j = 0;
                }
                it.next(p.seq_lens, p.B);
            }
            if (alive) {
                // the last segment: finish the older drain, capture, wait for its
                // last PV, write it out
                const int il = ntiles - 1;
                tc_fence_after();
                while (dr_left > 0) drain_step();
                capture(il + 1, seg);
                group_wait(&ctrl->o_done[il & 1], (il >> 1) & 1, p, ctrl, kSiteOFinal, il);
                named_bar_sync(1, 128);
                if (!ctrl->abort) {  // same value in every thread after the barrier
                    tc_fence_after();
                    start_drain(obuf, seg, il + 1, pend_b, pend_final);
                    while (dr_left > 0) drain_step();
                    if (st == 0) MLA_TRACE_POINT(il + 1, kTrEpiEnd);
                }
            }
            if (st == 0) MLA_KTRACE(2);
        }
    }
    __syncthreads();
    cluster_sync_all();  // no remote traffic into this CTA after here
    if (threadIdx.x == 0) MLA_KTRACE(3);
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ---------------------------------------------------------------- folded tiles
//
// Pools whose page size is a multiple of 8 rows: bf16 at 1..128 query rows,
// fp8_ds_mla at 1..64 (and bf16 rows of other latent widths). One CTA per
// worker, except the two cases below that pair two CTAs in a cluster. A tile
// is 64 tokens of whole rows,
// held as the 128-row A operand of one UMMA: row t (t < 64) carries token t's
// first half (latent [0, 256) and rope [512, 544)), row 64 + t its second half
// (latent [256, 512) and rope [544, 576)). With the query rows stacked the same
// way, B = [Q_a; Q_b] (N = 2 NP):
//   D[t, c]           = c_a(t) . q_a(c)   TMEM lanes 0..63,   columns [0, NP)
//   D[64 + t, NP + c] = c_b(t) . q_b(c)   TMEM lanes 64..127, columns [NP, 2 NP)
// so s(t, c) = D[t, c] + D[64 + t, NP + c]: the two halves of a token meet in
// shared memory between softmax warps 4/6 and 5/7, and each keeps half of the
// columns. (One 3-D TMA box per run carrying both halves halves the number of
// boxes, but measured slower: its loads land 2-4 us after issue, not ~1 us.)
// The value product reads the same tile as the MN-major A operand of four
// M = 128 UMMAs, K = 64 tokens; M-tile kb covers the latent dims of K-block kb
// in both halves, [64 kb, 64 kb + 64) and [256 + 64 kb, 256 + 64 kb + 64):
//   O^T[512, NP] += C^T[512, 64] . P[64, NP]
// so each 16-KB K-block is read by four S and four PV MMAs and nothing else,
// and the ring is in K-block slots that free one by one.
// Nothing crosses between CTAs: a tile's shared memory is held from its load
// to its value product only, with no exchange latency in between.
//
// Query rows: NP = 16, 32 or 64 a CTA. At 32 and 64 rows two softmax groups of
// four warps each own half of the columns (at 64 rows: half of the tile's
// tokens, for every query). At 64 rows the score product is transposed, with
// Q's latent part in TMEM as its A operand; the ring has eleven K-block slots
// and two rope slots, one S buffer, one P buffer and one O accumulator (a finished
// segment is written out before the next segment's first value product).
// 65..128 rows: the two 64-row groups of a worker run
// as a cluster of two CTAs that share each tile through multicast TMA (each
// issues half of the boxes into both), so the cache is read once per request.
// fp8_ds_mla rows: TMA lands each K-block's e4m3 codes in the upper half of
// its slot, four expand warps widen them in place to f16 (the queries' latent
// part and P are f16 too). Latent width 1792: the two latent halves of every row in the two
// CTAs of a cluster, which add their partial scores.

template <int NP, int KB, bool PAIR = false, int KIND = 0>
struct FoldCfg {
    static_assert(NP == 16 || NP == 32 || (NP == 64 && KB == 4 && !PAIR), "NP");
    // KIND 1: fp8_ds_mla rows (656 bytes) of the 576-wide row
    static_assert(KIND == 0 || (KB == 4 && !PAIR), "fp8 rows");
    // KB K-blocks per tile and CTA: 128 KB latent values in two halves of 64 KB.
    // PAIR: the two CTAs of a cluster take the latent's two halves (1792 = 2 x 896)
    static_assert(PAIR ? (KB == 7 && NP == 16) : (KB == 2 || KB == 4 || (KB == 6 && NP == 16)), "latent width");
    static constexpr int kDL = 128 * KB;                  // latent values this CTA holds
    static constexpr int kD = PAIR ? 2 * kDL : kDL;       // the row's latent width
    static constexpr int kHalf = 64 * KB;
    static constexpr int kTok = 64;                    // tokens per tile
    static constexpr int kBlkBytes = 128 * 128;        // a K-block: 64 dims x (64 + 64) rows, 128-B swizzled
    static constexpr int kRopeBytes = 128 * 64;        // 32 rope dims x 128 rows, 64-B swizzled
    // K-block slots (4 per tile) and rope slots (1 per tile, freed right after
    // S): at 32 rows a tenth K-block slot is worth more than a second rope slot
    // (the rope reload waits for one S, well inside a tile's time; 3% faster)
    // At 64 query rows only Q's rope part (8 KB) stays in shared memory: eleven
    // K-block slots (almost three tiles) and two rope slots fit beside one P
    // buffer and a half-width exchange buffer. With one rope slot, each
    // tile's rope copy would wait for the previous tile's score product, a
    // chain as long as a tile (twelve K-block slots and one rope slot: 2% slower).
    // kTr: at 64 rows the score product runs transposed, S^T = Q K^T, with the
    // latent part of Q as the A operand in TMEM (lanes 0..63: the queries'
    // first latent halves, 64..127: their second halves) and the tile as B, so
    // that Q's 64 KB leave shared memory for three more K-block slots and a
    // second rope slot. TMEM: O in columns [0, 256), Q in [256, 384), one S
    // buffer in [384, 512).
    // Latent width 768 (six K-blocks a tile, 16 rows): eleven K-block slots and
    // one rope slot (ten and two: 5% slower).
    static constexpr bool kTr = NP == 64;
    static constexpr int kRL = PAIR ? 9 : (KB == 4) ? ((NP == 16) ? 11 : NP == 32 ? 10 : 11)
                                                    : (KB == 2 ? ((NP == 16) ? 11 : 10) : (KB == 6 ? 11 : 10));
    static constexpr int kRR = (KB == 4) ? ((NP == 32) ? 1 : 2) : (KB == 6 ? 1 : 2);
    // K-blocks [kb_lo(pp), kb_hi(pp)) of each tile belong to producer pp and PV issuer pp
    static __host__ __device__ constexpr int kb_lo(int pp) { return pp ? (KB + 1) / 2 : 0; }
    static __host__ __device__ constexpr int kb_hi(int pp) { return pp ? KB : (KB + 1) / 2; }
    // Producer warp 1 fills, and PV issuer 0 frees, K-blocks 0 and 1 of each
    // tile; warp 8 and issuer 1 K-blocks 2 and 3, all in one ring. A producer
    // orders a refill only by its own earlier waits (and the rope slots it
    // shares with the other producer), and a parity wait cannot tell the
    // slot's last phase from the one before it; with 11 slots, or 10 and one
    // rope slot, those waits do prove the fill before last freed whichever
    // issuer runs behind (checked on a random-schedule model of the protocol).
    static __device__ __forceinline__ int slot_of(int i, int kb) { return (KB * i + kb) % kRL; }
    static __device__ __forceinline__ int fill_of(int i, int kb) { return (KB * i + kb) / kRL; }
    static constexpr int kQBytes = kTr ? 2 * NP * 64 : 2 * NP * (KB * 128 + 64);  // kTr: the rope part only
    // Softmax groups: at 32 and 64 rows of the 576-wide row two groups of four
    // warps, each owning half of the query columns (two warps per scheduler,
    // half the work per thread)
    static constexpr int kSG = (NP == 64 || (NP == 32 && KB == 4 && !PAIR)) ? 2 : 1;
    static constexpr int kGW = NP / kSG;               // columns per group
    static constexpr int kNH = kGW / 2;                // softmax columns per thread
    // the partner lane's half scores, kXR columns at a time (at 64 rows two
    // rounds of 8 per group, so the two groups' buffers take 8 KB; fp8 rows
    // four rounds of 4, measured faster there: the expand warps' registers)
    static constexpr int kXR = NP == 64 ? (KIND == 1 ? 4 : 8) : kNH;
    static constexpr int kXBytes = kSG * 128 * kXR * 4;
    // 9 warps, plus the second softmax group's 4
    // fp8 rows: four expand warps (one per K-block of a tile) widen the e4m3
    // codes into bf16; the pools' 64-token pages make few boxes a tile, so one
    // producer warp issues them all and the second producer warp is an
    // expander (four warps to a scheduler at most: 128 registers a thread)
    static constexpr int kExpandWarps = KIND == 1 ? 4 : 0;
    static constexpr int kProducers = KIND == 1 ? 1 : 2;
    static constexpr int kThreads = 288 + 128 * (kSG - 1) + 32 * (kExpandWarps - (kProducers == 1 ? 1 : 0));
    // K-blocks [kb_lo(pp), kb_hi(pp)) of each tile: producer pp (and PV issuer pp)
    static __host__ __device__ constexpr int prod_lo(int pp) { return kProducers == 1 ? 0 : kb_lo(pp); }
    static __host__ __device__ constexpr int prod_hi(int pp) { return kProducers == 1 ? KB : kb_hi(pp); }
    // one P buffer at 64 rows: the softmax writes P(i) once PV(i - 1) has
    // read P(i - 1), which a tile's softmax outlasts
    static constexpr int kPBufs = NP == 64 ? 1 : 2;
    static constexpr int kPBytes = kTok * NP * 2;      // P [64 tokens][NP] bf16, MN-major
    static constexpr int kOffRope = kRL * kBlkBytes;
    static constexpr int kOffQ = kOffRope + kRR * kRopeBytes;
    static constexpr int kOffX = (kOffQ + kQBytes + 1023) / 1024 * 1024;
    static constexpr int kOffP = kOffX + kXBytes;
    static constexpr int kX2Bytes = PAIR ? 128 * kNH * 4 : 0;  // the peer CTA's partial scores
    static constexpr int kOffX2 = kOffP + kPBufs * kPBytes;
    // fp8 rows: each tile's 64 rows of four fp32 block scales, in two slots
    // (tile i in slot i % 2)
    static constexpr int kScaleBytes = KIND == 1 ? kTok * 16 : 0;
    static constexpr int kOffScale = kOffX2 + kX2Bytes;
    static constexpr int kOffCtrl = kOffScale + 2 * kScaleBytes;
    static constexpr int kSmemBytes = kOffCtrl + 3584 + 1024;  // + control block, alignment slack
    // TMEM: two O accumulators of KB x NP columns (M-tile m at m * NP; one at
    // 64 rows, where two would leave no room for S), then two S buffers of
    // 2 x NP columns (at 64 rows: Q's latent part, then one S buffer). With
    // one accumulator a finished segment is drained before the next segment's
    // first value product.
    static constexpr bool kOneO = NP == 64;
    static constexpr int kColQ = KB * NP;               // kTr: Q's latent values, 2 a column
    static constexpr int kColS = kTr ? kColQ + 64 * KB / 2 : (kOneO ? 1 : 2) * KB * NP;
    static constexpr int kSBufs = kTr ? 1 : 2;
    static constexpr int kTmemCols = (kColS + kSBufs * 2 * NP) <= 128   ? 128
                                     : (kColS + kSBufs * 2 * NP) <= 256 ? 256
                                                                        : 512;
    // one row of P = one swizzle atom
    static constexpr uint32_t kPSwizzle = NP == 16 ? kSw32 : NP == 32 ? kSw64 : kSw128;
    static_assert(kSmemBytes <= 232448, "shared memory");
    static_assert(kColS + kSBufs * 2 * NP <= kTmemCols, "tmem");
};

struct FoldCtrl {
    uint64_t blk_full[12], blk_empty[12];
    uint64_t rope_full[2], rope_empty[2];
    uint64_t s_full[2], s_free[2], o_done[2], q_full;
    // tile t's P hand-off to the two PV issuers is p_full[t & 1]: the softmax
    // may hand over tile t + 1 as soon as PV(t - 1) is done, which can be
    // before a slow issuer has begun to wait for tile t, and one barrier would
    // then complete a phase past that issuer, whose parity wait could never
    // end; tile t + 2's hand-off follows PV(t) of both issuers
    uint64_t p_full[2];
    uint64_t x2full, x2free;         // CTA pair: the peer's partial scores landed / it has read ours
    uint64_t fin[3];                 // the S and PV issuers' products have all completed (at exit)
    uint64_t raw_full[12];           // fp8 rows: a K-block's codes landed in the upper half of its slot
    uint64_t q_tmem;                 // transposed scores: the softmax warps have written Q's latent part
    uint64_t scale_full[2], scale_empty[2];  // fp8 rows: a tile's block scales landed / both expanders done
    uint32_t tmem_base;
    int abort;
    int t_begin, t_end, b0, j0;
    int colvis[64];                  // uniform verify length: query row -> trailing tokens it may not see
    alignas(16) float m[64];         // running max per row (log2 units)
    alignas(16) float alpha[64];
    alignas(16) float red[4][64];    // per-warp column reductions
    alignas(16) float dlt[2][64];    // row sums of a finished segment, by segment parity
    float dm[2][64];                 // and its row maxima
};
static_assert(sizeof(FoldCtrl) <= 3584, "control block");

// MC: the two row groups of a worker (query rows 0..63 and 64..127 of each
// request) are the two CTAs of a cluster; each CTA loads half of every tile's
// boxes with multicast, so each cached row crosses HBM once for both groups,
// and a ring slot is refilled only when both CTAs' value products have
// released it.
// KIND 1: fp8_ds_mla rows. TMA lands each K-block's e4m3 codes in the upper
// half of its slot and each tile's block scales in a scale slot; two expand
// warps widen the codes into the bf16 layout the products read, in place.
template <int NP, int KB, bool PAIR, bool MC, int KIND>
__global__ void __launch_bounds__(FoldCfg<NP, KB, PAIR, KIND>::kThreads, 1)
    mla_decode_fold_kernel(const __grid_constant__ DecodeMaps maps, const DecodeParams p) {
    static_assert(!MC || (NP == 64 && !PAIR), "row-group pairs are 64-row CTAs");
    static_assert(!(MC && KIND == 1), "fp8 rows: one row group per worker");
    using C = FoldCfg<NP, KB, PAIR, KIND>;
    // first expand warp (fp8 rows), after the softmax groups
    constexpr int kExp0 = 9 + 4 * (C::kSG - 1);
    // the rope's element column in a row: after the latent (bf16), or at byte 528 (fp8)
    constexpr int kRopeX = KIND == 1 ? 264 : C::kD;
    constexpr uint16_t kPairMask = 0x3;
    constexpr int kT = C::kTok;
    using It = TileItT<6>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t* ring = smem;
    uint8_t* rope_ring = smem + C::kOffRope;
    uint8_t* qs = smem + C::kOffQ;
    uint8_t* xbuf = smem + C::kOffX;
    uint8_t* pbufs = smem + C::kOffP;
    uint8_t* x2buf = smem + C::kOffX2;
    uint8_t* scales = smem + C::kOffScale;
    FoldCtrl* ctrl = reinterpret_cast<FoldCtrl*>(smem + C::kOffCtrl);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // PAIR: a worker is a cluster of two CTAs, CTA r holding latent dims
    // [r kDL, (r + 1) kDL) of every row (and, r = 0 only, the rope)
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    const int g = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
    const int G = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
    const int gy = blockIdx.y;
    const int dbase = static_cast<int>(rank) * C::kDL;
    const bool has_rope = !PAIR || rank == 0;
    // MC: which half of every box pair (and which rope half) this CTA issues
    const int mrank = MC ? static_cast<int>(cluster_ctarank()) : 0;
    if (threadIdx.x == 0) MLA_KTRACE(0);

    if (threadIdx.x == 0) {
        // MC: a slot is released by the value products of both CTAs
        for (int i = 0; i < C::kRL; ++i) {
            mbar_init(&ctrl->blk_full[i], 1);
            mbar_init(&ctrl->blk_empty[i], MC ? 2 : 1);
        }
        // a rope slot is armed by both producer warps (one half each)
        for (int i = 0; i < C::kRR; ++i) {
            mbar_init(&ctrl->rope_full[i], C::kProducers);
            mbar_init(&ctrl->rope_empty[i], MC ? 2 : 1);
        }
        for (int i = 0; i < 3; ++i) mbar_init(&ctrl->fin[i], 1);
        if constexpr (KIND == 1) {
            for (int i = 0; i < C::kRL; ++i) mbar_init(&ctrl->raw_full[i], 1);
            for (int i = 0; i < 2; ++i) {
                mbar_init(&ctrl->scale_full[i], 1);
                mbar_init(&ctrl->scale_empty[i], C::kExpandWarps);
            }
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctrl->s_full[i], 1);
            mbar_init(&ctrl->s_free[i], C::kSG);  // one arrive per softmax group
            mbar_init(&ctrl->o_done[i], 2);  // one commit per PV issuer
        }
        mbar_init(&ctrl->q_tmem, 4 * C::kSG);  // one arrive per softmax warp
        mbar_init(&ctrl->p_full[0], C::kSG);
        mbar_init(&ctrl->p_full[1], C::kSG);
        mbar_init(&ctrl->q_full, 1);
        mbar_init(&ctrl->x2full, 1);  // + the peer's st.async bytes
        mbar_init(&ctrl->x2free, 1);  // the peer's remote arrive
        ctrl->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1 && lane == 0) {
        prefetch_tensormap(&maps.lat);
        prefetch_tensormap(&maps.rope);
        prefetch_tensormap(&maps.q);
        prefetch_tensormap(&maps.qpe);
    }
    // the previous kernel in the stream may still be writing the inputs or
    // reading the workspace
    griddep_wait();
    if (threadIdx.x == 0) {
        int4* r = reinterpret_cast<int4*>(status_rec(p));
#pragma unroll
        for (int k = 0; k < kStatusRecWords / 4; ++k) r[k] = make_int4(0, 0, 0, 0);
    }
    if (warp == 0) {
        tmem_alloc(&ctrl->tmem_base, C::kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    if (warp == 2) {
        const TileRange r = scan_range<6>(p, g, G, lane);
        if (lane == 0) {
            ctrl->t_begin = r.tb;
            ctrl->t_end = r.te;
            ctrl->b0 = r.b0;
            ctrl->j0 = r.j0;
        }
    }
    if (threadIdx.x >= 128 && threadIdx.x < 128 + 64) {
        const int c = threadIdx.x - 128;
        const int r = gy * 64 + c;
        ctrl->colvis[c] = (r < p.HQ) ? (p.Qt - 1 - r / p.Hq) : (INT_MAX / 2);
        ctrl->m[c] = -INFINITY;
    }
    __syncthreads();
    if constexpr (PAIR || MC) cluster_sync_all();  // the peer's barriers exist before any remote traffic
    if (threadIdx.x == 0) {
        MLA_KTRACE(1);
#ifdef MLA_TRACE
        unsigned sm;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
        MLA_KSM(0, sm);
        MLA_KSM(1, ctrl->t_end - ctrl->t_begin);
#endif
        griddep_launch_dependents();  // the merge grid may be scheduled as CTAs retire
    }
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    const int ntiles = ctrl->t_end - ctrl->t_begin;
    if (has_rope && ntiles == 0 && ctrl->j0 > 0 && threadIdx.x >= 128 && threadIdx.x < 192) {
        // an empty range strictly inside request b0 (more workers than tiles):
        // the merge of b0 counts this worker's slot, so mark it empty
        const int64_t pslot = static_cast<int64_t>(gy) * p.SPG + g + ctrl->b0;
        p.part_lse[pslot * 64 + (threadIdx.x - 128)] = -INFINITY;
    }

    if (ntiles > 0) {
        if (warp == 0 && lane == 0) {
            // -------------------------------------------------- S issuer
            // The rope's two products come first and release the rope slot with
            // a commit of their own: the producers load tile i + 1's rope as soon
            // as S(i) has read this one, and with one rope slot a release at the
            // end of S(i) would chain every tile's rope copy behind the previous
            // tile's whole score product.
            It it;
            it.init(p.seq_lens, ctrl->b0, ctrl->j0);
            const uint32_t idS = idesc_bf16(128, 2 * NP, false, false);
            // fp8 rows: the latent products are f16 (the widened cache, Q in TMEM)
            const uint32_t idSlat = idesc_bf16(128, 2 * NP, false, false, KIND == 1);
            const uint64_t dq = smem_desc(smem_u32(qs), 16, 1024, kSw128);
            const uint64_t dqr = smem_desc(smem_u32(qs) + (C::kTr ? 0 : 2 * KB * NP * 128), 16, 512, kSw64);
            int seg = 0;
            for (int i = 0; i < ntiles; ++i) {
                if (i == 0 || it.j == 0) {
                    // a new request: its Q (with kTr, the rope part here and the
                    // latent part in TMEM, written by the softmax warps)
                    if (!mbar_wait(&ctrl->q_full, seg & 1, &ctrl->abort) ||
                        ((C::kTr || KIND == 1) && !mbar_wait(&ctrl->q_tmem, seg & 1, &ctrl->abort))) {
                        fail(p, ctrl, kErrWaitTimeout, kSiteQFull, i);
                        report(p, kRoleS, kSiteQFull, i);
                        break;
                    }
                    ++seg;
                }
                // the softmax has read S(i - kSBufs) from the buffer S(i) writes
                if (i >= C::kSBufs &&
                    !mbar_wait(&ctrl->s_free[i % C::kSBufs], ((i / C::kSBufs) - 1) & 1, &ctrl->abort)) {
                    fail(p, ctrl, kErrWaitTimeout, kSiteSFree, i);
                    report(p, kRoleS, kSiteSFree, i);
                    break;
                }
                const uint32_t tS = tmem + C::kColS + (i % C::kSBufs) * 2 * NP;
                bool ok = true;
                int site = kSitePairFull;
                const int rr = i % C::kRR;
                if (has_rope) {
                    if (!mbar_wait(&ctrl->rope_full[rr], (i / C::kRR) & 1, &ctrl->abort)) {
                        ok = false;
                        site = kSiteRopeFull;
                    } else {
                        tc_fence_after();
                        MLA_TRACE_POINT(i, kTrSRope);
                        const uint64_t dr = smem_desc(smem_u32(rope_ring + rr * C::kRopeBytes), 16, 512, kSw64);
                        if constexpr (C::kTr) {
                            umma_bf16(tS, dqr, dr, idS, 0u);
                            umma_bf16(tS, dqr + 2, dr + 2, idS, 1u);
                        } else {
                            umma_bf16(tS, dr, dqr, idS, 0u);
                            umma_bf16(tS, dr + 2, dqr + 2, idS, 1u);
                        }
                        if constexpr (MC) umma_commit_mc(&ctrl->rope_empty[rr], kPairMask);
                        else umma_commit(&ctrl->rope_empty[rr]);
                    }
                }
                for (int kb = 0; kb < KB && ok; ++kb) {
                    const int slot = C::slot_of(i, kb);
                    if (!mbar_wait(&ctrl->blk_full[slot], C::fill_of(i, kb) & 1, &ctrl->abort)) { ok = false; break; }
                    tc_fence_after();
                    if (kb == 0) MLA_TRACE_POINT(i, kTrSPair0);
                    else if (kb < 4) MLA_TRACE_POINT(i, kTrSKb1 + kb - 1);
                    const uint64_t da = smem_desc(smem_u32(ring + slot * C::kBlkBytes), 16, 1024, kSw128);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        if constexpr (C::kTr)
                            umma_bf16_ta(tS, tmem + C::kColQ + kb * 32 + kk * 8, da + ((kk * 32) >> 4), idSlat, 1u);
                        else
                            umma_bf16(tS, da + ((kk * 32) >> 4), dq + ((kb * 2 * NP * 128 + kk * 32) >> 4),
                                      KIND == 1 ? idSlat : idS, (has_rope || (kb | kk) != 0) ? 1u : 0u);
                    }
                }
                if (!ok) {
                    fail(p, ctrl, kErrWaitTimeout, site, i);
                    report(p, kRoleS, site, i);
                    break;
                }
                MLA_TRACE_POINT(i, kTrSAllIn);
                umma_commit(&ctrl->s_full[i % C::kSBufs]);
                MLA_TRACE_POINT(i, kTrSIssued);
                it.next(p.seq_lens, p.B);
            }
            // every product issued here completes before the CTA may release
            // TMEM or exit (on the abort path some are still running)
            drain_mma(&ctrl->fin[0]);
        } else if ((warp == 3 || warp == 2) && lane == 0) {
            // ------------------------------------------------- PV issuers
            // issuer mt takes K-blocks 2 mt and 2 mt + 1: M-tile kb reads K-block
            // kb's slot as C^T (its two 64-dim atoms are the halves, 8 KB apart)
            // and frees the slot when its four MMAs are done
            const int mt = warp == 3 ? 0 : 1;
            It it;
            it.init(p.seq_lens, ctrl->b0, ctrl->j0);
            // P: [64 tokens][NP] (MN-major), or with kTr [NP queries][64 tokens]
            // (K-major, a 128-byte row per query)
            const uint32_t idPV = idesc_bf16(128, NP, true, !C::kTr, KIND == 1);
            constexpr uint32_t p_sbo = 8 * NP * 2;

            int seg = -1;
            for (int i = 0; i < ntiles; ++i) {
                const bool new_seg = (i == 0) || (it.j == 0);
                if (new_seg) ++seg;
                const uint32_t tO = tmem + (C::kOneO ? 0 : (seg & 1) * KB * NP);
                if (!mbar_wait(&ctrl->p_full[i & 1], (i >> 1) & 1, &ctrl->abort)) {
                    fail(p, ctrl, kErrWaitTimeout, kSitePFull, i);
                    report(p, kRolePV, kSitePFull, i);
                    break;
                }
                tc_fence_after();
                if (mt == 0) MLA_TRACE_POINT(i, kTrPvIssue);
                const uint64_t dp = C::kTr ? smem_desc(smem_u32(pbufs + (i % C::kPBufs) * C::kPBytes), 16, 1024, kSw128)
                                           : smem_desc(smem_u32(pbufs + (i % C::kPBufs) * C::kPBytes), C::kPBytes,
                                                       p_sbo, C::kPSwizzle);
#pragma unroll
                for (int q = 0; q < (KB + 1) / 2; ++q) {
                    const int kb = C::kb_lo(mt) + q;
                    if (kb >= C::kb_hi(mt)) break;
                    const int slot = C::slot_of(i, kb);
                    // tokens 16 kk .. 16 kk + 15: rows 16 kk .. of both halves
                    const uint64_t da = smem_desc(smem_u32(ring + slot * C::kBlkBytes), 8192, 1024, kSw128);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        umma_bf16(tO + kb * NP, da + ((kk * 2048) >> 4),
                                  dp + ((C::kTr ? kk * 32 : kk * 16 * NP * 2) >> 4), idPV,
                                  (new_seg && kk == 0) ? 0u : 1u);
                    if constexpr (MC) umma_commit_mc(&ctrl->blk_empty[slot], kPairMask);
                    else umma_commit(&ctrl->blk_empty[slot]);
                }
                umma_commit(&ctrl->o_done[i & 1]);
                if (p.test_hold == 2 && mt == 1 && i < 32) spin_for_ns(20000);  // test hook: a lagging issuer
                if (mt == 0) MLA_TRACE_POINT(i, kTrPvIssued);
                it.next(p.seq_lens, p.B);
            }
            drain_mma(&ctrl->fin[1 + mt]);
        } else if (warp == 1 || (warp == 8 && C::kProducers == 2)) {
            // ------------------------------------------------- TMA producers
            // Warp 1 loads K-blocks 0, 1 and the first rope half of every tile,
            // warp 8 K-blocks 2, 3 and the second rope half (with 16-token pages a
            // tile is 40 boxes of 2 KB, and one warp issuing them all takes about
            // as long as the tile's compute). Lane r owns run r of the tile (a
            // page-contiguous run of BR rows); each run lands twice per K-block:
            // its first halves in rows [r BR, (r+1) BR), its second halves 64
            // rows further. Page numbers are read one tile ahead.
            const int pp = warp == 1 ? 0 : 1;
            It it;
            it.init(p.seq_lens, ctrl->b0, ctrl->j0);
            const uint64_t pol = l2_policy_evict_first();
            const int BR = p.run_rows;
            bool bad = false, ok = true;
            int fsite = 0, ftile = 0;
            auto run_slot = [&](const It& t) -> int {
                const int valid = min(kT, t.T - t.j * kT);
                const int nr = (valid + BR - 1) / BR;
                const int32_t* btr = p.block_table + static_cast<int64_t>(t.b) * p.bt_stride;
                return lane < nr ? static_cast<int>(token_slot(p, btr, t.j * kT + lane * BR, bad)) : 0;
            };
            int y_next = run_slot(it);
            // K-block fills (tile-major, this warp's K-blocks) and rope fills (tiles)
            // whose barriers this warp has armed: at exit it waits for those fills
            // to land, so that no copy arrives after the CTA is gone
            int armed = 0, rope_armed = 0, scale_armed = 0;
            for (int i = 0; i < ntiles && ok; ++i) {
                const int valid = min(kT, it.T - it.j * kT);
                const int nruns = (valid + BR - 1) / BR;
                const int y = y_next;
                const uint32_t run_bytes = static_cast<uint32_t>(nruns * BR * 128);
                It nx = it;
                nx.next(p.seq_lens, p.B);
                if (i + 1 < ntiles) y_next = run_slot(nx);
                if (lane == 0) MLA_TRACE_POINT(i, pp ? kTrProd1Start : kTrProdStart);
                if (has_rope) {
                    const int rr = i % C::kRR;
                    if (i >= C::kRR &&
                        !__all_sync(0xffffffffu, mbar_wait(&ctrl->rope_empty[rr], ((i / C::kRR) - 1) & 1, &ctrl->abort))) {
                        ok = false;
                        fsite = kSiteTmaRopeEmpty;
                        ftile = i;
                        break;
                    }
                    if (lane == 0 && pp == 0) MLA_TRACE_POINT(i, kTrEpiStored);  // rope slot free
                    // rope half pp (each producer one half; a single producer both),
                    // before the tile's K-blocks: its slot comes free first
                    if (lane == 0) mbar_arrive_expect_tx(&ctrl->rope_full[rr], C::kProducers == 1 ? run_bytes : run_bytes / 2);
                    __syncwarp();
                    rope_armed = i + 1;
                    if constexpr (C::kProducers == 1) {
                        if (lane < nruns) {
#pragma unroll
                            for (int rh = 0; rh < 2; ++rh)
                                tma_load_2d(rope_ring + rr * C::kRopeBytes + rh * 4096 + lane * BR * 64, &maps.rope,
                                            &ctrl->rope_full[rr], kRopeX + 32 * rh, y, pol);
                        }
                    } else if (lane < nruns) {
                        if constexpr (MC) {
                            // rope half pp comes from the CTA of rank pp, into both CTAs
                            if (pp == mrank)
                                tma_load_2d_mc(rope_ring + rr * C::kRopeBytes + pp * 4096 + lane * BR * 64, &maps.rope,
                                               &ctrl->rope_full[rr], kRopeX + 32 * pp, y, kPairMask, pol);
                        } else {
                            tma_load_2d(rope_ring + rr * C::kRopeBytes + pp * 4096 + lane * BR * 64, &maps.rope,
                                        &ctrl->rope_full[rr], kRopeX + 32 * pp, y, pol);
                        }
                    }
                    if (lane == 0 && pp == 0) MLA_TRACE_POINT(i, kTrProdIssued);
                }
                for (int q = 0; q < C::prod_hi(pp) - C::prod_lo(pp); ++q) {
                    const int kb = C::prod_lo(pp) + q;
                    const int slot = C::slot_of(i, kb), fill = C::fill_of(i, kb);
                    if (fill > 0 &&
                        !__all_sync(0xffffffffu, mbar_wait(&ctrl->blk_empty[slot], (fill - 1) & 1, &ctrl->abort))) {
                        ok = false;
                        fsite = kSiteTmaPairEmpty;
                        ftile = i;
                        break;
                    }
                    if (lane == 0 && q == 0) MLA_TRACE_POINT(i, kTrEpiStart + pp);  // slot free
                    if constexpr (MC) {
                        // a peer that has given up may leave at any time: send it nothing more
                        if (__shfl_sync(0xffffffffu, lane == 0 ? peer_aborted(&ctrl->abort, mrank ^ 1) : 0, 0)) {
                            ok = false;
                            fsite = kSiteTmaPairEmpty;
                            ftile = i;
                            break;
                        }
                    }
                    if constexpr (KIND == 1) {
                        // the codes of both halves (64 bytes a row each) into the slot's
                        // upper half: first-half rows at 8 KB, second-half rows at 12 KB
                        if (lane == 0) mbar_arrive_expect_tx(&ctrl->raw_full[slot], 2u * nruns * BR * 64);
                        __syncwarp();
                        if (lane < nruns) {
                            uint8_t* dst = ring + slot * C::kBlkBytes + 8192 + lane * BR * 64;
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh)
                                tma_load_2d(dst + hh * 4096, &maps.lat, &ctrl->raw_full[slot], 256 * hh + 64 * kb, y,
                                            pol);
                        }
                        armed = i * (C::prod_hi(pp) - C::prod_lo(pp)) + q + 1;
                        continue;
                    }
                    if (lane == 0) mbar_arrive_expect_tx(&ctrl->blk_full[slot], 2 * run_bytes);
                    __syncwarp();
                    if (lane < nruns) {
                        uint8_t* dst = ring + slot * C::kBlkBytes + lane * BR * 128;
                        if constexpr (MC) {
                            // this CTA's half of the pair, into both CTAs
                            const int hh = mrank;
                            tma_load_2d_mc(dst + hh * 8192, &maps.lat, &ctrl->blk_full[slot], C::kHalf * hh + 64 * kb, y,
                                           kPairMask, pol);
                        } else {
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh)
                                tma_load_2d(dst + hh * 8192, &maps.lat, &ctrl->blk_full[slot],
                                            dbase + C::kHalf * hh + 64 * kb, y, pol);
                        }
                    }
                    armed = i * (C::prod_hi(pp) - C::prod_lo(pp)) + q + 1;
                }
                if (!ok) break;
                if (lane == 0) MLA_TRACE_POINT(i, pp ? kTrProd1Done : kTrProd0Done);
                if constexpr (KIND == 1) {
                    if (pp == 0) {
                        // the tile's block scales, 16 bytes a row, once both expanders
                        // are done with the slot's tile before last
                        const int sb = i & 1;
                        if (i >= 2 &&
                            !__all_sync(0xffffffffu, mbar_wait(&ctrl->scale_empty[sb], ((i >> 1) - 1) & 1, &ctrl->abort))) {
                            ok = false;
                            fsite = kSiteRawFull;
                            ftile = i;
                            break;
                        }
                        if (lane == 0) mbar_arrive_expect_tx(&ctrl->scale_full[sb], static_cast<uint32_t>(nruns * BR * 16));
                        __syncwarp();
                        scale_armed = i + 1;
                        if (lane < nruns)
                            tma_load_2d(scales + sb * C::kScaleBytes + lane * BR * 16, &maps.aux, &ctrl->scale_full[sb], 512,
                                        y, pol);
                    }
                }
                it = nx;
            }
            if (!ok && lane == 0) {
                fail(p, ctrl, kErrWaitTimeout, fsite, ftile);
                report(p, pp ? kRoleLsu0 : kRoleTma, fsite, ftile);  // no load/convert warps here: their slot
            }
            if (lane == 0 && ctrl->abort) {
                // Abort path: copies this warp armed may still be in flight; let them
                // land before the CTA leaves (on the normal path every fill has been
                // consumed by S). The last fill of each slot this warp armed, newest
                // first; a slot the other producer refilled later (a shared ring)
                // cannot be told apart by parity and waits out the deadline, which
                // is one for all of them.
                volatile int never = 0;
                const unsigned long long t0 = globaltimer_ns();
                const int nk = C::prod_hi(pp) - C::prod_lo(pp);
                uint32_t seen = 0;
                for (int a = armed - 1; a >= 0 && a >= armed - 2 * C::kRL; --a) {
                    const int t = a / nk, kb = C::prod_lo(pp) + a % nk;
                    const int slot = C::slot_of(t, kb);
                    if (seen & (1u << slot)) continue;
                    seen |= 1u << slot;
                    uint64_t* full = KIND == 1 ? &ctrl->raw_full[slot] : &ctrl->blk_full[slot];
                    while (!mbar_try_wait(full, C::fill_of(t, kb) & 1) && !never && globaltimer_ns() - t0 < kWaitLimitNs) {
                    }
                }
                for (int t = scale_armed - 1; t >= 0 && t >= scale_armed - 2; --t)
                    while (!mbar_try_wait(&ctrl->scale_full[t & 1], (t >> 1) & 1) && !never &&
                           globaltimer_ns() - t0 < kWaitLimitNs) {
                    }
                seen = 0;
                for (int t = rope_armed - 1; t >= 0 && t >= rope_armed - 4; --t) {
                    const int rr = t % C::kRR;
                    if (seen & (1u << rr)) continue;
                    seen |= 1u << rr;
                    while (!mbar_try_wait(&ctrl->rope_full[rr], (t / C::kRR) & 1) && !never &&
                           globaltimer_ns() - t0 < kWaitLimitNs) {
                    }
                }
            }
            if (bad) atomicOr(status_rec(p), kErrBadBlock);
        } else if (KIND == 1 && (warp >= kExp0 || warp == 8)) {
            // ------------------------------------------- expand warps (fp8 rows)
            // Warp e widens K-block e of every tile: the codes TMA
            // landed in the upper half of the slot (first-half rows at 8 KB + 64 t,
            // second-half rows at 12 KB + 64 t for token t) become rows of the
            // 128-byte-swizzled layout S and PV read, each code times its token's
            // scale of the 128-value block it belongs to, in f16: the code exact
            // in f16, one f16 multiply rounded to nearest even, two instructions
            // for two values where a bf16 result takes six (f16 holds every such
            // product more precisely than bf16; a scale above kMaxF16Scale, which
            // could overflow it, is reported in the status word). The queries'
            // latent part (in TMEM at 64 rows, converted in place in shared
            // memory at 16 and 32) and P are f16 as well; the rope stays bf16. A
            // second-half row overwrites codes, so every lane holds its codes in
            // registers before any row is written.
            const int e = warp == 8 ? 0 : warp - kExp0 + 1;  // K-block e of every tile
            bool ok = true;
            int fsite = 0, ftile = 0;
            It it;  // the tile's request: rows past its end hold stale bytes, not checked
            it.init(p.seq_lens, ctrl->b0, ctrl->j0);
            for (int i = 0; i < ntiles && ok; ++i) {
                const int sb = i & 1;
                const int valid = min(kT, it.T - it.j * kT);
                if (!mbar_wait(&ctrl->scale_full[sb], (i >> 1) & 1, &ctrl->abort)) {
                    ok = false;
                    fsite = kSiteRawFull;
                    ftile = i;
                    break;
                }
                const uint8_t* sc = scales + sb * C::kScaleBytes;
                for (int q = 0; q < KB / (C::kExpandWarps > 0 ? C::kExpandWarps : 1); ++q) {
                    const int kb = e + q;
                    const int slot = C::slot_of(i, kb);
                    if (!mbar_wait(&ctrl->raw_full[slot], C::fill_of(i, kb) & 1, &ctrl->abort)) {
                        ok = false;
                        fsite = kSiteRawFull;
                        ftile = i;
                        break;
                    }
                    if (lane == 0 && e == 0 && q == 0) MLA_TRACE_POINT(i, kTrSmXFree);  // codes landed
                    uint8_t* blk = ring + slot * C::kBlkBytes;
                    // Lane l takes a quarter (16 codes, 32 bf16 bytes) of row 8 it + l / 4
                    // in each of eight steps: a warp-wide 16-byte load then covers 512
                    // contiguous code bytes (no bank conflicts), and the two stores of
                    // a step hit every bank group once.
                    const int uq = lane & 3;
                    bool wide = false;  // a scale past the f16 range
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        // the step's codes and scales all in flight at once (a scale
                        // read after the previous step's stores would wait for them:
                        // the compiler cannot tell the two regions apart)
                        uint4 cd[8];
                        float scl[8];
#pragma unroll
                        for (int it = 0; it < 8; ++it) {
                            cd[it] = *reinterpret_cast<const uint4*>(blk + 8192 + h * 4096 + it * 512 + lane * 16);
                            scl[it] = *reinterpret_cast<const float*>(sc + (8 * it + (lane >> 2)) * 16 + 4 * (2 * h + (kb >> 1)));
                        }
                        __syncwarp();  // every lane's codes are in registers
#pragma unroll
                        for (int it = 0; it < 8; ++it) {
                            const int t = 8 * it + (lane >> 2), r = 64 * h + t;
                            uint4 lo, hi;
                            wide |= t < valid && !(scl[it] <= kMaxF16Scale);
                            dequant16_h(cd[it], __float2half2_rn(scl[it]), lo, hi);
                            uint8_t* row = blk + r * 128;
                            *reinterpret_cast<uint4*>(row + (((2 * uq) ^ (r & 7)) << 4)) = lo;
                            *reinterpret_cast<uint4*>(row + (((2 * uq + 1) ^ (r & 7)) << 4)) = hi;
                        }
                        __syncwarp();  // the first halves' codes are consumed before h = 1 writes over them
                    }
                    if (__any_sync(0xffffffffu, wide) && lane == 0) atomicOr(status_rec(p), kErrF16Range);
                    fence_proxy_async_smem();  // the products read these rows through the async proxy
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ctrl->blk_full[slot]);
                }
                if (!ok) break;
                it.next(p.seq_lens, p.B);
                if (lane == 0) mbar_arrive(&ctrl->scale_empty[sb]);
                if (lane == 0) MLA_TRACE_POINT(i, e == 0 ? kTrEpiEnd : kTrEpiHalf);  // expander e done with tile i
            }
            if (!ok && lane == 0) {
                fail(p, ctrl, kErrWaitTimeout, fsite, ftile);
                report(p, kRoleLsu0 + 1, fsite, ftile);
            }
        } else if ((warp >= 4 && warp < 8) || (warp >= 9 && warp < kExp0)) {
            // ------------------------------------------ softmax + epilogue
            // Thread st reads TMEM lane st = A row st: half hf of token tt (lane
            // quadrants 0, 1 the first halves, 2, 3 the second). Softmax group grp
            // (warps 4..7, and at 64 rows 9..12) owns query columns [cg0, cg0 +
            // GW): the thread keeps [own0, own0 + NH) and hands the group's other
            // NH partial scores to its partner st ^ 64, the other half of the same
            // token.
            // kTr (64 rows, S^T): lane st holds half hf of query tt's scores and
            // the columns are the tile's token halves, so the same exchange leaves
            // the thread the whole scores of query tt for tokens [own0, own0 +
            // NH); the four threads of a query (two halves, two groups) meet for
            // its row maximum and sum, and O's columns stay the groups' queries.
            const int grp = warp >= 9 ? 1 : 0;
            const int sw = warp & 3;  // TMEM lane quadrant
            const int st = sw * 32 + lane;
            const int hf = sw >> 1;
            const int tt = st & 63;
            const uint32_t lane_base = static_cast<uint32_t>(sw * 32) << 16;
            constexpr int NH = C::kNH, GW = C::kGW;
            const int cg0 = grp * GW;
            const int own0 = cg0 + hf * NH;
            const int par0 = cg0 + (hf ? 0 : NH);  // the partner's columns
            const int bsync = grp ? 3 : 1, bvote = grp ? 4 : 2;  // the group's named barriers
            constexpr int kBarAll = 5, kBarAllOr = 6;             // both groups (kTr)
            const bool lead = grp == 0 && st == 0;  // once-per-CTA work of the tile
            // exchange rows of XR floats (the group's own rows), 16-byte units
            // swizzled by row; thread st writes row st ^ 64 and reads row st (same
            // swizzle: bit 6 is not in it)
            constexpr int XR = C::kXR;
            uint8_t* xg = xbuf + grp * 128 * XR * 4;
            const int xs = (XR == 16) ? ((st >> 1) & 3) : (XR == 8) ? ((st >> 2) & 1) : 0;
            It it;
            it.init(p.seq_lens, ctrl->b0, ctrl->j0);
            // the current segment's verify length and its rows in this row group
            int seg_qt = req_qt(p, it.b), seg_hq = req_rows_in_group(p, it.b, gy);
            float l[NH];
#pragma unroll
            for (int c = 0; c < NH; ++c) l[c] = 0.f;
            int seg_start_j = it.j;
            bool seg_has_pv = false;
            int seg = 0;
            uint32_t obuf = 0;
            bool pend = false, pend_final = false;
            int pend_b = 0;
            int dr_left = 0, dr_step = 0, dr_b = 0, dr_sg = 0;
            bool dr_final = false;
            uint32_t dr_obuf = 0;
            constexpr int kDC = 8;  // columns per drain step
            int dr_hq = 0, dr_per_mt = 1;  // rows of the segment being drained (in this row group)
            int64_t dr_row0 = 0;           // and its first output row

            // Column reductions over the tile's tokens: a warp reduces its 32
            // lanes (one half), red[warp][column] meets the other warps' (the
            // identity in the columns of the half the warp does not hold).
            auto red_store = [&](int c, float v, float ident) {
                if (lane == 0) {
                    ctrl->red[sw][own0 + c] = v;
                    ctrl->red[sw][par0 + c] = ident;
                }
            };

            // O columns [cg0, cg0 + GW) of accumulator ob, all M-tiles, times
            // alpha (the caller has waited for the last PV into it)
            auto rescale_o = [&](uint32_t ob) {
                tc_fence_after();
                __syncwarp();
#pragma unroll 1
                for (int m4 = 0; m4 < KB; ++m4)
#pragma unroll 1
                    for (int c0 = cg0; c0 < cg0 + GW; c0 += 16) {
                        uint32_t o[16];
                        tmem_ld_x16(tmem + lane_base + ob + m4 * NP + c0, o);
#pragma unroll
                        for (int cc = 0; cc < 16; ++cc)
                            o[cc] = __float_as_uint(__uint_as_float(o[cc]) * ctrl->alpha[c0 + cc]);
                        tmem_st_x16(tmem + lane_base + ob + m4 * NP + c0, o);
                    }
                tmem_wait_st();
            };

            // The NP query rows of request bq (row group gy) by TMA, stacked as
            // S reads them: K-block k holds rows [0, NP) = latent dims 64k.. and
            // rows [NP, 2NP) = dims 256 + 64k.. (128-B swizzle, at k * 2NP * 128),
            // then the rope halves (64-B swizzle, at 8 NP * 128).
            auto issue_q = [&](int bq) {
                const int y = static_cast<int>(req_row0(p, bq) + gy * 64);
                const uint64_t pol = l2_policy_evict_first();
                mbar_arrive_expect_tx(&ctrl->q_full, has_rope ? C::kQBytes : C::kQBytes - 2 * NP * 64);
                if constexpr (!C::kTr) {
#pragma unroll
                    for (int k = 0; k < KB; ++k)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh)
                            tma_load_2d(qs + (k * 2 + hh) * NP * 128, &maps.q, &ctrl->q_full,
                                        dbase + C::kHalf * hh + 64 * k, y, pol);
                }
                if (has_rope) {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh)
                        tma_load_2d(qs + (C::kTr ? 0 : 2 * KB * NP * 128) + hh * NP * 64, &maps.qpe, &ctrl->q_full,
                                    32 * hh, y, pol);
                }
            };

            // kTr: Q's latent part of request bq into TMEM, the A operand of S^T:
            // lane st holds half hf of query tt (latent dims 256 hf ..), group grp
            // its columns [64 grp, 64 grp + 64) (dims 256 hf + 128 grp ..); padding
            // rows are zeros. Called once S has read the previous request's Q.
            auto write_q = [&](int bq) {
                const bool v = tt < req_rows_in_group(p, bq, gy);
                const __nv_bfloat16* src =
                    p.q_lat + (req_row0(p, bq) + gy * 64 + (v ? tt : 0)) * static_cast<int64_t>(C::kD) + 256 * hf + 128 * grp;
                bool wide = false;  // fp8 rows: a value past the f16 range
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t r[16];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint4 w = v ? __ldg(reinterpret_cast<const uint4*>(src + 32 * q4 + 8 * u)) : make_uint4(0, 0, 0, 0);
                        r[4 * u] = w.x;
                        r[4 * u + 1] = w.y;
                        r[4 * u + 2] = w.z;
                        r[4 * u + 3] = w.w;
                    }
                    if constexpr (KIND == 1) {
                        // the cache side is f16 here, so Q's latent part is too (every
                        // bf16 value in the f16 range converts exactly)
#pragma unroll
                        for (int k = 0; k < 16; ++k) {
                            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&r[k]));
                            wide |= !(fabsf(f.x) <= 65504.f) || !(fabsf(f.y) <= 65504.f);
                            r[k] = pack_half2(f.x, f.y);
                        }
                    }
                    tmem_st_x16(tmem + lane_base + C::kColQ + 64 * grp + 16 * q4, r);
                }
                if (KIND == 1 && __any_sync(0xffffffffu, wide) && lane == 0) atomicOr(status_rec(p), kErrF16Range);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctrl->q_tmem);
            };

            // fp8 rows at 16 and 32 rows: once the request's queries have landed
            // in shared memory (bf16), their latent part becomes f16 in place, the
            // type of the widened cache; the rope part stays bf16.
            int qseg = 0;
            auto convert_q = [&]() {
                group_wait(&ctrl->q_full, qseg & 1, p, ctrl, kSiteQFull, 0);
                ++qseg;
                constexpr int kUnits = 2 * NP * KB * 128 / 16;  // 16-byte units of the latent part
                bool wide = false;
                for (int u = grp * 128 + st; u < kUnits; u += 128 * C::kSG) {
                    uint4* q = reinterpret_cast<uint4*>(qs) + u;
                    uint4 w = *q;
                    uint32_t* e = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&e[k]));
                        wide |= !(fabsf(f.x) <= 65504.f) || !(fabsf(f.y) <= 65504.f);
                        e[k] = pack_half2(f.x, f.y);
                    }
                    *q = w;
                }
                if (__any_sync(0xffffffffu, wide) && lane == 0) atomicOr(status_rec(p), kErrF16Range);
                fence_proxy_async_smem();  // the score product reads them through the async proxy
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctrl->q_tmem);
            };

            // Row sums and maxima of segment sg, which just ended, into
            // dlt / dm [sg & 1]; fresh softmax state for the next segment.
            auto capture = [&](int sg) {
                if constexpr (C::kTr) {
                    // query tt's sum: this thread's tokens, the partner half's, the
                    // other group's two
                    ctrl->red[2 * grp + hf][tt] = l[0];
                    named_bar_sync(kBarAll, 256);
                } else {
#pragma unroll
                    for (int c = 0; c < NH; ++c) red_store(c, warp_sum(l[c]), 0.f);
                    named_bar_sync(bsync, 128);
                }
                if (st < GW) {
                    const int c = cg0 + st;
                    ctrl->dlt[sg & 1][c] = ctrl->red[0][c] + ctrl->red[1][c] + ctrl->red[2][c] + ctrl->red[3][c];
                    ctrl->dm[sg & 1][c] = ctrl->m[c];
                    ctrl->m[c] = -INFINITY;
                }
#pragma unroll
                for (int c = 0; c < NH; ++c) l[c] = 0.f;
                if constexpr (C::kTr) named_bar_sync(kBarAll, 256);
                else named_bar_sync(bsync, 128);
            };

            // The captured segment sg (accumulator src) has had its last PV:
            // write its LSEs and start draining its rows.
            auto start_drain = [&](uint32_t src, int sg, int sb, bool sfinal, int shq) {
                const int64_t pslot = static_cast<int64_t>(gy) * p.SPG + g + sb;
                dr_row0 = req_row0(p, sb) + gy * 64;
                if (st < GW && cg0 + st < shq && rank == 0) {
                    const int c = cg0 + st;
                    const float lt = ctrl->dlt[sg & 1][c];
                    const float lv = lt > 0.f ? (ctrl->dm[sg & 1][c] + log2f(lt)) * kLn2 : -INFINITY;
                    if (sfinal) p.lse[dr_row0 + c] = lv;
                    else p.part_lse[pslot * 64 + c] = lv;
                }
                dr_hq = shq;
                const int gq = min(GW, max(0, shq - cg0));  // the segment's rows in this group's columns
                dr_per_mt = max(1, (gq + kDC - 1) / kDC);
                dr_left = gq > 0 ? KB * dr_per_mt : 0;
                dr_step = 0;
                dr_b = sb;
                dr_final = sfinal;
                dr_obuf = src;
                dr_sg = sg;
                pend = false;
            };

            // One drain step: kDC columns of one M-tile, O / l, into the output
            // rows (a whole request) or this worker's partial slot. A thread's TMEM
            // lane is one latent dim; each quad of lanes transposes 4 x 4 blocks so
            // that a lane stores 4 consecutive dims of one row in one 16-byte store
            // (one-value stores made the drain ~6x slower).
            auto drain_step = [&]() {
                const int m4 = dr_step / dr_per_mt;
                const int c0 = cg0 + (dr_step - m4 * dr_per_mt) * kDC;
                uint32_t o[kDC];
                tmem_ld_x8(tmem + lane_base + dr_obuf + m4 * NP + c0, o);
                // M-tile m4, lane st: latent dim 64 m4 + st (first half) or 256 + 64 m4 + st - 64;
                // the quad's first dim
                const int64_t dq = dbase + (st < 64 ? 0 : C::kHalf - 64) + 64 * m4 + (st & ~3);
                const int64_t pslot = static_cast<int64_t>(gy) * p.SPG + g + dr_b;
                if constexpr (KIND == 1 && C::kTr) {
                    // fp8 rows at 64 rows: one value a store (the transpose's registers
                    // cost that kernel more than the stores, measured 2%)
                    const int64_t d = dq + (st & 3);
#pragma unroll
                    for (int cc = 0; cc < kDC; ++cc) {
                        const int c = c0 + cc;
                        if (c < dr_hq) {
                            const float lt = ctrl->dlt[dr_sg & 1][c];
                            const float v = lt > 0.f ? __uint_as_float(o[cc]) / lt : 0.f;
                            if (dr_final) {
                                const int64_t idx = (dr_row0 + c) * C::kD + d;
                                if (p.out_f32) static_cast<float*>(p.out)[idx] = v;
                                else static_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(v);
                            } else {
                                p.part_o[(pslot * 64 + c) * C::kD + d] = v;
                            }
                        }
                    }
                } else {
#pragma unroll
                    for (int cb = 0; cb < kDC; cb += 4) {
                        float x[4] = {__uint_as_float(o[cb]), __uint_as_float(o[cb + 1]), __uint_as_float(o[cb + 2]),
                                      __uint_as_float(o[cb + 3])};
                        quad_transpose(x, lane);
                        const int c = c0 + cb + (lane & 3);  // this lane's row now
                        if (c < dr_hq) {
                            const float lt = ctrl->dlt[dr_sg & 1][c];
                            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (lt > 0.f) v = make_float4(x[0] / lt, x[1] / lt, x[2] / lt, x[3] / lt);
                            if (dr_final) {
                                const int64_t idx = (dr_row0 + c) * C::kD + dq;
                                if (p.out_f32)
                                    *reinterpret_cast<float4*>(static_cast<float*>(p.out) + idx) = v;
                                else
                                    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + idx) =
                                        make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
                            } else {
                                *reinterpret_cast<float4*>(p.part_o + (pslot * 64 + c) * C::kD + dq) = v;
                            }
                        }
                    }
                }
                ++dr_step;
                --dr_left;
            };

            int cap_b = 0, cap_hq = 0;
            bool cap_final = false;

            // Hand tile t to the PV issuers, then start or advance the drain.
            // False when the group aborts.
            auto finish = [&](int t, bool aborted) -> bool {
                if (aborted) return false;  // the same value in every thread of the group (kTr: of both)
                if (st == 0) {
                    // (one arrive per group) the test hook withholds tile 0, so the PV
                    // issuers' bounded wait gives up and every role leaves through the
                    // abort path
                    if (lead) {
                        MLA_TRACE_POINT(t, kTrSmPArrive);
                        MLA_TTRACE(t);
                    }
                    if (!(p.test_hold == 1 && t == 0)) mbar_arrive(&ctrl->p_full[t & 1]);
                }
                seg_has_pv = true;
                if (pend) {
                    // PV(t-1), the captured segment's last, is long done by now
                    group_wait(&ctrl->o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, p, ctrl, kSiteOEpi, t);
                    tc_fence_after();
                    start_drain(obuf ^ (KB * NP), seg - 1, cap_b, cap_final, cap_hq);
                } else if (dr_left > 0) {
                    tc_fence_after();
                    drain_step();
                    tc_fence_before();
                }
                return true;
            };

            if (lead) issue_q(it.b);
            if constexpr (C::kTr) write_q(it.b);
            else if constexpr (KIND == 1) convert_q();
            bool alive = true;
            for (int i = 0; i < ntiles; ++i) {
                const int b = it.b, j = it.j, T = it.T;
                const bool last_of_seg = (j == it.tiles - 1) || (i == ntiles - 1);
                group_wait(&ctrl->s_full[i % C::kSBufs], (i / C::kSBufs) & 1, p, ctrl, kSiteSFull, i);
                if (lead) MLA_TRACE_POINT(i, kTrSmSFull);
                if (lead && last_of_seg && i + 1 < ntiles) {
                    // S(i) is complete, so Q may be replaced by the next request's
                    It nx = it;
                    nx.next(p.seq_lens, p.B);
                    issue_q(nx.b);
                }
                tc_fence_after();
                __syncwarp();
                // this lane's half of the scores: the group's columns of [hf NP, hf NP +
                // NP) (a TMEM load takes one column address per warp: hf is the same
                // in the warp). It keeps the NH columns [own0, own0 + NH) and writes
                // the other NH into its partner's exchange row, XR at a time.
                const uint32_t s_addr = tmem + lane_base + C::kColS + (i % C::kSBufs) * 2 * NP + hf * NP + cg0;
                uint32_t sr[GW];
                tmem_ld_np<GW>(s_addr, sr);
                tc_fence_before();
                uint32_t own[NH];
                // compile-time indices so sr[] stays in registers
#pragma unroll
                for (int k = 0; k < NH; ++k) own[k] = hf ? sr[NH + k] : sr[k];
                auto snd = [&](int k) -> uint32_t { return hf ? sr[k] : sr[NH + k]; };
                // partner columns [base, base + XR) into exchange row st ^ 64
                auto put_x = [&](int base) {
#pragma unroll
                    for (int u = 0; u < XR / 4; ++u)
                        *reinterpret_cast<uint4*>(xg + (st ^ 64) * XR * 4 + ((u ^ xs) << 4)) =
                            make_uint4(snd(base + 4 * u), snd(base + 4 * u + 1), snd(base + 4 * u + 2),
                                       snd(base + 4 * u + 3));
                };
                put_x(0);
                if (lead) MLA_TRACE_POINT(i, kTrSmTmemLd);
                if (KIND == 1 && lead && (i == 0 || j == 0) && !last_of_seg) {
                    // fp8 rows: warm L2 with the next request's queries and page list
                    // (measured: 2% for fp8 pools; no gain elsewhere, where its loads
                    // stall the group at request boundaries)
                    It nx = it;
                    nx.j = nx.tiles - 1;
                    nx.next(p.seq_lens, p.B);
                    if (nx.b < p.B) prefetch_request(p, nx.b, gy);
                }
                if (lead) MLA_TRACE_POINT(i, kTrSmSent);
                if (i > 0 && j == 0) {
                    // the previous segment ended with tile i-1: finish the older
                    // drain (its accumulator is the one this segment will use)
                    if (dr_left > 0) {
                        tc_fence_after();
                        while (dr_left > 0) drain_step();
                        tc_fence_before();
                    }
                    capture(seg);  // its barriers also order the exchange rows
                    if constexpr (C::kOneO) {
                        // one accumulator: the ended segment's O (its last value product
                        // is PV(i - 1)) is written out before PV(i) may start this one
                        group_wait(&ctrl->o_done[(i - 1) & 1], ((i - 1) >> 1) & 1, p, ctrl, kSiteOEpi, i);
                        tc_fence_after();
                        if (!ctrl->abort) {
                            start_drain(0u, seg, pend_b, pend_final, seg_hq);
                            while (dr_left > 0) drain_step();
                        }
                        tc_fence_before();
                    } else {
                        pend = true;
                        cap_b = pend_b;
                        cap_final = pend_final;
                        cap_hq = seg_hq;
                    }
                    seg_qt = req_qt(p, b);
                    seg_hq = req_rows_in_group(p, b, gy);
                    seg_has_pv = false;
                    ++seg;
                    obuf = C::kOneO ? 0u : static_cast<uint32_t>((seg & 1) * KB * NP);
                } else {
                    named_bar_sync(bsync, 128);
                }
                if (st == 0) mbar_arrive(&ctrl->s_free[i % C::kSBufs]);  // every thread of the group has read S(i)
                if (lead) MLA_TRACE_POINT(i, kTrSmXFull);
                float x[NH];
                // own columns [base, base + XR) plus the partner's half of them
                auto read_x = [&](int base) {
#pragma unroll
                    for (int u = 0; u < XR / 4; ++u) {
                        const float4 v = *reinterpret_cast<const float4*>(xg + st * XR * 4 + ((u ^ xs) << 4));
                        x[base + 4 * u] = __uint_as_float(own[base + 4 * u]) + v.x;
                        x[base + 4 * u + 1] = __uint_as_float(own[base + 4 * u + 1]) + v.y;
                        x[base + 4 * u + 2] = __uint_as_float(own[base + 4 * u + 2]) + v.z;
                        x[base + 4 * u + 3] = __uint_as_float(own[base + 4 * u + 3]) + v.w;
                    }
                };
                read_x(0);
#pragma unroll
                for (int r = XR; r < NH; r += XR) {
                    named_bar_sync(bsync, 128);  // every thread has read the last round
                    put_x(r);
                    named_bar_sync(bsync, 128);
                    read_x(r);
                }
                if constexpr (PAIR) {
                    // the other CTA of the pair holds the other latent half: add its
                    // partial scores of this thread's token and columns (row st of
                    // each CTA's x2buf, written by st.async), then hand the buffer
                    // back once every thread has read it. Both CTAs add the same two
                    // values, so their scores, and every softmax decision, agree.
                    const uint32_t peer = rank ^ 1u;
                    if (i > 0) group_wait(&ctrl->x2free, (i - 1) & 1, p, ctrl, kSiteXFree, i, true);
                    if (st == 0) mbar_arrive_expect_tx(&ctrl->x2full, C::kX2Bytes);
                    const uint32_t dst = mapa_shared(smem_u32(x2buf + st * NH * 4), peer);
                    const uint32_t bar = mapa_shared(smem_u32(&ctrl->x2full), peer);
#pragma unroll
                    for (int u = 0; u < NH / 4; ++u)
                        st_async_v4(dst + 16 * u, __float_as_uint(x[4 * u]), __float_as_uint(x[4 * u + 1]),
                                    __float_as_uint(x[4 * u + 2]), __float_as_uint(x[4 * u + 3]), bar);
                    group_wait(&ctrl->x2full, i & 1, p, ctrl, kSiteXFull, i, true);
#pragma unroll
                    for (int u = 0; u < NH / 4; ++u) {
                        const float4 v = *reinterpret_cast<const float4*>(x2buf + st * NH * 4 + 16 * u);
                        x[4 * u] += v.x;
                        x[4 * u + 1] += v.y;
                        x[4 * u + 2] += v.z;
                        x[4 * u + 3] += v.w;
                    }
                    named_bar_sync(bsync, 128);
                    if (st == 0) mbar_arrive_remote_relaxed(mapa_shared(smem_u32(&ctrl->x2free), peer));
                }
                if (lead) MLA_TRACE_POINT(i, kTrSmXRead);
                const int tok = j * kT + tt;
                const bool all_vis = (j * kT + kT + seg_qt - 1) <= T;
                const float4* m4p = reinterpret_cast<const float4*>(ctrl->m + own0);
                if constexpr (C::kTr) {
                    // x[c]: query tt, token j kT + own0 + c
                    if (all_vis) {
                        const bool qv = tt < seg_hq;
#pragma unroll
                        for (int c = 0; c < NH; ++c) x[c] = qv ? x[c] * p.scale_log2 : -INFINITY;
                    } else if (p.cu_q) {
                        const int r = gy * 64 + tt;
                        const int lim = T - (seg_qt - 1 - r / p.Hq) - (j * kT + own0);  // visible: c < lim
                        const bool qv = tt < seg_hq;
#pragma unroll
                        for (int c = 0; c < NH; ++c) x[c] = (qv && c < lim) ? x[c] * p.scale_log2 : -INFINITY;
                    } else {
                        const int lim = T - ctrl->colvis[tt] - (j * kT + own0);
#pragma unroll
                        for (int c = 0; c < NH; ++c) x[c] = (c < lim) ? x[c] * p.scale_log2 : -INFINITY;
                    }
                } else if (all_vis) {
#pragma unroll
                    for (int c = 0; c < NH; ++c) x[c] = (own0 + c < seg_hq) ? x[c] * p.scale_log2 : -INFINITY;
                } else {
                    // tail of a request: query token r / Hq of the step sees tokens up to
                    // T - Qt + r / Hq, and rows past the request's are padding
                    if (p.cu_q) {
#pragma unroll
                        for (int c = 0; c < NH; ++c) {
                            const int r = gy * 64 + own0 + c;
                            const bool v = own0 + c < seg_hq && tok + seg_qt - 1 - r / p.Hq < T;
                            x[c] = v ? x[c] * p.scale_log2 : -INFINITY;
                        }
                    } else {
                        // the same limits, tabulated once (every request has p.Qt tokens)
#pragma unroll
                        for (int c = 0; c < NH; ++c)
                            x[c] = (tok + ctrl->colvis[own0 + c] < T) ? x[c] * p.scale_log2 : -INFINITY;
                    }
                }
                int need = 0;
                if constexpr (C::kTr) {
                    const float mq = ctrl->m[tt] + kRescaleThreshold;
#pragma unroll
                    for (int c = 0; c < NH; ++c) need |= x[c] > mq;
                } else {
#pragma unroll
                    for (int u = 0; u < NH / 4; ++u) {
                        const float4 mv = m4p[u];
                        need |= (x[4 * u] > mv.x + kRescaleThreshold) | (x[4 * u + 1] > mv.y + kRescaleThreshold) |
                                (x[4 * u + 2] > mv.z + kRescaleThreshold) | (x[4 * u + 3] > mv.w + kRescaleThreshold);
                    }
                }
                // (also: every thread has read its exchange row)
                if (lead) MLA_TRACE_POINT(i, kTrSmMath);
                // kTr: a query's maximum involves both groups, and so does its O column
                need = C::kTr ? named_bar_or(kBarAllOr, 256, need) : named_bar_or(bvote, 128, need);
                if (lead) MLA_TRACE_POINT(i, kTrSmBarOr);
                if (need && C::kTr) {
                    // query tt's maximum over the tile: its four threads' maxima
                    float mx = x[0];
#pragma unroll
                    for (int c = 1; c < NH; ++c) mx = fmaxf(mx, x[c]);
                    ctrl->red[2 * grp + hf][tt] = mx;
                    named_bar_sync(kBarAll, 256);
                    if (grp == 0 && hf == 0) {
                        const float mt = fmaxf(fmaxf(ctrl->red[0][tt], ctrl->red[1][tt]), fmaxf(ctrl->red[2][tt], ctrl->red[3][tt]));
                        const float mo = ctrl->m[tt];
                        const float mn = fmaxf(mo, mt);
                        ctrl->alpha[tt] = (mo == -INFINITY) ? 0.f : ex2(mo - mn);
                        ctrl->m[tt] = mn;
                    }
                    named_bar_sync(kBarAll, 256);
                    l[0] *= ctrl->alpha[tt];
                    if (seg_has_pv) {
                        group_wait(&ctrl->o_done[(i - 1) & 1], ((i - 1) >> 1) & 1, p, ctrl, kSiteORescale, i);
                        rescale_o(obuf);
                        if (lead) MLA_TRACE_POINT(i, kTrSmRescaled);
                    }
                } else if (need) {
                    // column maxima over the tile's 64 tokens
#pragma unroll
                    for (int c = 0; c < NH; ++c) red_store(c, warp_max(x[c]), -INFINITY);
                    named_bar_sync(bsync, 128);
                    if (st < GW) {
                        const int c = cg0 + st;
                        const float mt = fmaxf(fmaxf(ctrl->red[0][c], ctrl->red[1][c]), fmaxf(ctrl->red[2][c], ctrl->red[3][c]));
                        const float mo = ctrl->m[c];
                        const float mn = fmaxf(mo, mt);
                        ctrl->alpha[c] = (mo == -INFINITY) ? 0.f : ex2(mo - mn);
                        ctrl->m[c] = mn;
                    }
                    named_bar_sync(bsync, 128);
#pragma unroll
                    for (int c = 0; c < NH; ++c) l[c] *= ctrl->alpha[own0 + c];
                    if (seg_has_pv) {
                        // O holds earlier tiles of this segment: wait for their PV, rescale
                        // every column (each thread its TMEM lane of the four M-tiles)
                        group_wait(&ctrl->o_done[(i - 1) & 1], ((i - 1) >> 1) & 1, p, ctrl, kSiteORescale, i);
                        rescale_o(obuf);
                        if (lead) MLA_TRACE_POINT(i, kTrSmRescaled);
                    }
                }
                if constexpr (C::kTr) {
                    const float mq = ctrl->m[tt];
                    const float mk = (mq == -INFINITY) ? 0.f : mq;
                    float ls = 0.f;
#pragma unroll
                    for (int c = 0; c < NH; ++c) {
                        x[c] = ex2(x[c] - mk);
                        ls += x[c];
                    }
                    l[0] += ls;
                } else {
#pragma unroll
                    for (int u = 0; u < NH / 4; ++u) {
                        const float4 mv = m4p[u];
                        const float mm[4] = {mv.x, mv.y, mv.z, mv.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int c = 4 * u + k;
                            const float mk = (mm[k] == -INFINITY) ? 0.f : mm[k];
                            const float pc = ex2(x[c] - mk);
                            l[c] += pc;
                            x[c] = pc;
                        }
                    }
                }
                if (lead) MLA_TRACE_POINT(i, kTrSmExpLoop);
                // the P buffer of this tile was last read by PV(i - kPBufs)
                if (i >= C::kPBufs) {
                    const int jp = i - C::kPBufs;
                    bool okp = true;
                    if (lane == 0) okp = !ctrl->abort && mbar_wait(&ctrl->o_done[jp & 1], (jp >> 1) & 1, &ctrl->abort);
                    okp = __shfl_sync(0xffffffffu, okp ? 1 : 0, 0) != 0;
                    if (!okp && lane == 0) fail(p, ctrl, kErrWaitTimeout, kSiteOPbuf, i);
                }
                if (lead) MLA_TRACE_POINT(i, kTrSmExp);
                // P row tt, columns [own0, own0 + NH): NH / 8 16-byte units (kTr: row
                // = query tt, columns = tokens: the K-major P the value product reads)
                const int pb = i % C::kPBufs;
                uint8_t* prow = pbufs + pb * C::kPBytes + tt * NP * 2;
                const int sz = swz_p(tt, C::kPSwizzle);
#pragma unroll
                for (int u = 0; u < NH / 8; ++u) {
                    const int un = own0 / 8 + u;
                    const uint4 v = KIND == 1
                                        ? make_uint4(pack_half2(x[8 * u + 0], x[8 * u + 1]), pack_half2(x[8 * u + 2], x[8 * u + 3]),
                                                           pack_half2(x[8 * u + 4], x[8 * u + 5]), pack_half2(x[8 * u + 6], x[8 * u + 7]))
                                              : make_uint4(pack_bf16x2(x[8 * u + 0], x[8 * u + 1]), pack_bf16x2(x[8 * u + 2], x[8 * u + 3]),
                                                           pack_bf16x2(x[8 * u + 4], x[8 * u + 5]), pack_bf16x2(x[8 * u + 6], x[8 * u + 7]));
                    *reinterpret_cast<uint4*>(prow + ((un ^ sz) << 4)) = v;
                }
                if (grp == 0 && j * kT + tt >= T) {
                    // this row's token is past the request: its bytes are stale (maybe
                    // NaN); P is 0 there, but 0 * NaN would still poison O, so clear
                    // the row in the four K-blocks (rotated units: no bank conflicts)
                    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                    for (int q = 0; q < KB; ++q) {
                        uint8_t* row = ring + C::slot_of(i, q) * C::kBlkBytes + st * 128;
#pragma unroll
                        for (int u = 0; u < 8; ++u) *reinterpret_cast<uint4*>(row + (((u + st) & 7) << 4)) = z;
                    }
                }
                if (lead) MLA_TRACE_POINT(i, kTrSmPStore);
                fence_proxy_async_smem();
                tc_fence_before();
                // kTr: the groups meet at barriers of all 256 threads, so they must
                // leave together: the abort flag is read in one reduction
                bool aborted;
                if constexpr (C::kTr) {
                    aborted = named_bar_or(kBarAllOr, 256, ctrl->abort != 0) != 0;
                } else {
                    named_bar_sync(bsync, 128);
                    aborted = ctrl->abort != 0;
                }
                if (!finish(i, aborted)) {
                    alive = false;
                    break;
                }
                if (last_of_seg) {
                    pend_final = (seg_start_j == 0) && (j == it.tiles - 1);
                    pend_b = b;
                    seg_start_j = 0;
                }
                it.next(p.seq_lens, p.B);
                // S(i), the request's last score product, has read Q: the next one's
                if (C::kTr && last_of_seg && i + 1 < ntiles) write_q(it.b);
                if (!C::kTr && KIND == 1 && last_of_seg && i + 1 < ntiles) convert_q();
            }
            if (alive) {
                // the last segment: finish the older drain, capture, wait for its
                // last PV, write it out
                const int il = ntiles - 1;
                tc_fence_after();
                while (dr_left > 0) drain_step();
                capture(seg);
                group_wait(&ctrl->o_done[il & 1], (il >> 1) & 1, p, ctrl, kSiteOFinal, il);
                named_bar_sync(bsync, 128);
                if (!ctrl->abort) {
                    tc_fence_after();
                    start_drain(obuf, seg, pend_b, pend_final, seg_hq);
                    while (dr_left > 0) drain_step();
                }
            }
            if (st == 0) MLA_KTRACE(2);
        }
    }
    __syncthreads();
    if constexpr (PAIR || MC) cluster_sync_all();  // no remote traffic into this CTA after here
    if (threadIdx.x == 0) MLA_KTRACE(3);
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

// ---------------------------------------------------------------- merging

// Merge `nseg` partials of one row: out = sum_i w_i o_i with
// w_i = exp(lse_i - L), L = ln sum exp(lse_i); all -inf -> (0, -inf).
// One warp; lane owns dims 4*lane + 128*k, k = 0..3.
__device__ __forceinline__ void merge_row(const float* po, int64_t o_stride, const float* pl, int64_t l_stride,
                                          int nseg, void* out, int out_f32, float* lse_out, int lane) {
    float mx = -INFINITY;
    for (int s = lane; s < nseg; s += 32) mx = fmaxf(mx, pl[s * l_stride]);
    mx = warp_max(mx);
    float4 acc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = -INFINITY;
    if (mx != -INFINITY) {
        float ws = 0.f;
        for (int s = lane; s < nseg; s += 32) {
            const float v = pl[s * l_stride];
            if (v != -INFINITY) ws += expf(v - mx);
        }
        ws = warp_sum(ws);
        L = mx + logf(ws);
        for (int s = 0; s < nseg; ++s) {
            const float v = pl[s * l_stride];
            if (v == -INFINITY) continue;
            const float w = expf(v - L);
            const float4* src = reinterpret_cast<const float4*>(po + s * o_stride);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 o = src[lane + 32 * k];
                acc[k].x += w * o.x;
                acc[k].y += w * o.y;
                acc[k].z += w * o.z;
                acc[k].w += w * o.w;
            }
        }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int d = 4 * lane + 128 * k;
        if (out_f32) {
            reinterpret_cast<float4*>(static_cast<float*>(out) + d)[0] = acc[k];
        } else {
            __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(out) + d;
            reinterpret_cast<uint2*>(ob)[0] = make_uint2(pack_bf16x2(acc[k].x, acc[k].y), pack_bf16x2(acc[k].z, acc[k].w));
        }
    }
    if (lane == 0 && lse_out) *lse_out = L;
}

// Decode merge: RPB rows of one request per block, GRP groups of 128 threads
// per row; thread t of group grp holds dims 4t .. 4t+3 of the row's partial
// slots k = grp (mod GRP), and the groups' sums meet in shared memory (GRP = 4
// when rows have dozens of slots, 1 otherwise). Rows of requests that one
// worker held whole were written by the decode kernel; rows of requests cut
// across workers g0..g1 combine their partial slots g + b; rows of empty
// requests get (0, -inf). Block (0, 0) also folds the per-CTA status records
// of the decode grid into the workspace header.
// VP float4 columns per thread: thread t of a row owns dims 4t + 512v, v < VP,
// below the latent width (VP = 2 for 768).
template <int RPB, int GRP, int VP>
__global__ void __launch_bounds__(128 * RPB * GRP) mla_decode_merge_kernel(const DecodeParams p, int G, int nrec) {
    constexpr int kThreads = 128 * RPB * GRP;
    const int64_t D = p.lat_dim;
    MLA_MTRACE(0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int RB = (min(64, p.HQ) + RPB - 1) / RPB;  // blocks per (request, row group)
    const int b = blockIdx.x / RB, gy = blockIdx.y;
    const int rb = tid / (128 * GRP);
    const int n = (blockIdx.x - b * RB) * RPB + rb;
    const int t = tid & 127, grp = (tid >> 7) % GRP;
    // cost coordinate of request b's first tile, and the total cost (the
    // decode kernel's work split)
    __shared__ long long red_pre[kThreads / 32], red_tot[kThreads / 32];
    __shared__ float4 part[GRP > 1 ? GRP - 1 : 1][VP][128];
    long long pre = 0, tot = 0;
    for (int i = tid; i < p.B; i += kThreads) {
        const long long tl = (max(__ldg(p.seq_lens + i), 0) + (1 << p.tile_shift) - 1) >> p.tile_shift;
        const long long c = tl > 0 ? tl + p.wseg : 0;
        tot += c;
        if (i < b) pre += c;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        pre += __shfl_xor_sync(0xffffffffu, pre, o);
        tot += __shfl_xor_sync(0xffffffffu, tot, o);
    }
    if (lane == 0) { red_pre[warp] = pre; red_tot[warp] = tot; }
    __syncthreads();
    pre = p.wseg;
    tot = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) { pre += red_pre[w]; tot += red_tot[w]; }
    griddep_wait();  // the decode grid has finished and its writes are visible

    if (blockIdx.x == 0 && blockIdx.y == 0 && warp == 0) {
        // status summary: OR of all records; the lowest failing CTA's site,
        // tile, index and role reports
        int bits = 0, first = INT_MAX;
#pragma unroll 8
        for (int c = lane; c < nrec; c += 32) {  // independent loads, in flight together
            const int v = p.rec[static_cast<int64_t>(c) * kStatusRecWords];
            bits |= v;
            if (v && c < first) first = c;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            bits |= __shfl_xor_sync(0xffffffffu, bits, o);
            first = min(first, __shfl_xor_sync(0xffffffffu, first, o));
        }
        if (lane < 16) {
            int v = 0;
            if (lane == 0) v = bits;
            else if (first != INT_MAX) {
                const int* r = p.rec + static_cast<int64_t>(first) * kStatusRecWords;
                v = lane == 1 ? r[1] : lane == 2 ? r[2] : lane == 3 ? first : (lane < 12 ? r[lane] : 0);
            }
            p.status[lane] = v;
        }
    }

    if (b >= p.B) return;
    if (n >= req_rows_in_group(p, b, gy)) return;  // the same for the whole block when it holds one row
    const int tiles_b = (max(__ldg(p.seq_lens + b), 0) + (1 << p.tile_shift) - 1) >> p.tile_shift;
    const int64_t row = req_row0(p, b) + gy * 64 + n;
    const int d = 4 * t;
    bool dv[VP];
#pragma unroll
    for (int v = 0; v < VP; ++v) dv[v] = d + 512 * v < D;
    float4 acc[VP];
#pragma unroll
    for (int v = 0; v < VP; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = -INFINITY;
    if (tiles_b > 0) {
        // the workers holding the first and last tile: the largest g with
        // floor(g * tot / G) <= cost coordinate of the tile
        const long long g0 = ((pre + 1) * G - 1) / tot;
        const long long g1 = ((pre + tiles_b) * G - 1) / tot;
        if (g0 == g1) return;  // one worker held the whole request and wrote the output
        const int nseg = static_cast<int>(g1 - g0 + 1);
        const int64_t slot0 = static_cast<int64_t>(gy) * p.SPG + g0 + b;
        const float* pl = p.part_lse + slot0 * 64 + n;
        const float* po = p.part_o + (slot0 * 64 + n) * D + d;
        // this group's slots k = grp, grp + GRP, ...: the first kSpec of them are
        // requested before the weights are known, so the loads overlap the LSE
        // round trip (empty slots hold stale values and get weight 0)
        constexpr int kSpec = GRP > 1 ? 4 : 8;
        const int nmine = nseg > grp ? (nseg - grp + GRP - 1) / GRP : 0;
        float4 ov[kSpec][VP];
#pragma unroll
        for (int k = 0; k < kSpec; ++k)
#pragma unroll
            for (int v = 0; v < VP; ++v)
                if (k < nmine && dv[v])
                    ov[k][v] = *reinterpret_cast<const float4*>(po + static_cast<int64_t>(grp + GRP * k) * 64 * D + 512 * v);
        // the slot LSEs, 32 at a time, one per lane (every warp computes the
        // same weights)
        float mx = -INFINITY;
        for (int c0 = 0; c0 < nseg; c0 += 32)
            mx = fmaxf(mx, c0 + lane < nseg ? pl[(c0 + lane) * 64] : -INFINITY);
        mx = warp_max(mx);
        if (mx != -INFINITY) {
            float ws = 0.f;
            for (int c0 = 0; c0 < nseg; c0 += 32) {
                const float v = c0 + lane < nseg ? pl[(c0 + lane) * 64] : -INFINITY;
                ws += v != -INFINITY ? expf(v - mx) : 0.f;
            }
            L = mx + logf(warp_sum(ws));
            auto add = [&](int k, const float4 (&o)[VP]) {
                const float lv = pl[k * 64];
                const float w = lv != -INFINITY ? expf(lv - L) : 0.f;
                if (w != 0.f) {
#pragma unroll
                    for (int v = 0; v < VP; ++v) {
                        if (!dv[v]) continue;
                        acc[v].x += w * o[v].x;
                        acc[v].y += w * o[v].y;
                        acc[v].z += w * o[v].z;
                        acc[v].w += w * o[v].w;
                    }
                }
            };
#pragma unroll
            for (int k = 0; k < kSpec; ++k)
                if (k < nmine) add(grp + GRP * k, ov[k]);
            // the rest, 8 loads in flight at a time
            for (int k0 = kSpec; k0 < nmine; k0 += 8) {
                float4 o8[8][VP];
#pragma unroll
                for (int k = 0; k < 8; ++k)
#pragma unroll
                    for (int v = 0; v < VP; ++v)
                        if (k0 + k < nmine && dv[v])
                            o8[k][v] = *reinterpret_cast<const float4*>(
                                po + static_cast<int64_t>(grp + GRP * (k0 + k)) * 64 * D + 512 * v);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    if (k0 + k < nmine) add(grp + GRP * (k0 + k), o8[k]);
            }
        }
    }
    if constexpr (GRP > 1) {
        // the groups' sums (every group has L; the empty-request path too). The
        // block has one row, so every return above was taken by all of it.
        if (grp > 0) {
#pragma unroll
            for (int v = 0; v < VP; ++v) part[grp - 1][v][t] = acc[v];
        }
        __syncthreads();
        if (grp > 0) return;
#pragma unroll
        for (int q = 0; q < GRP - 1; ++q)
#pragma unroll
            for (int v = 0; v < VP; ++v) {
                const float4 o = part[q][v][t];
                acc[v].x += o.x;
                acc[v].y += o.y;
                acc[v].z += o.z;
                acc[v].w += o.w;
            }
    }
#pragma unroll
    for (int v = 0; v < VP; ++v) {
        if (!dv[v]) continue;
        if (p.out_f32) {
            *reinterpret_cast<float4*>(static_cast<float*>(p.out) + row * D + d + 512 * v) = acc[v];
        } else {
            *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.out) + row * D + d + 512 * v) =
                make_uint2(pack_bf16x2(acc[v].x, acc[v].y), pack_bf16x2(acc[v].z, acc[v].w));
        }
    }
    if (t == 0) p.lse[row] = L;
    MLA_MTRACE(1);
}

// Public split-KV combine: part_o [S, N, 512], part_lse [S, N]. One warp per row.
__global__ void __launch_bounds__(256) mla_merge_lse_kernel(const float* __restrict__ part_o,
                                                            const float* __restrict__ part_lse, int S, int64_t N,
                                                            void* out, int out_f32, float* lse) {
    const int64_t n = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (n >= N) return;
    merge_row(part_o + n * kD, N * kD, part_lse + n, N, S,
              static_cast<uint8_t*>(out) + n * kD * (out_f32 ? 4 : 2), out_f32, lse ? lse + n : nullptr,
              threadIdx.x & 31);
}

// ------------------------------------------------------------------ launch

// Launch configuration that lets the grid start while the previous kernel
// in the stream drains (the kernel calls griddep_wait() before touching
// global memory that kernel may use).
static cudaLaunchConfig_t pdl_config(dim3 grid, int threads, size_t smem, cudaStream_t stream,
                                     cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// The merge grid for G workers: rows whose requests are cut into dozens of
// slots (workers >= 8 per request) get four thread groups each; otherwise two
// rows share a block of one group each.
static cudaError_t launch_decode_merge(const DecodeParams& p, int G, int nrec, int GY, cudaStream_t stream) {
    const bool wide = G >= 8 * p.B;
    const int rows = min(64, p.HQ);
    const int RB = wide ? rows : (rows + 1) / 2;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg =
        pdl_config(dim3(static_cast<unsigned>(p.B) * RB, GY), wide ? 512 : 256, 0, stream, attr);
    if (p.lat_dim > 1024)
        return wide ? cudaLaunchKernelEx(&cfg, mla_decode_merge_kernel<1, 4, 4>, p, G, nrec)
                    : cudaLaunchKernelEx(&cfg, mla_decode_merge_kernel<2, 1, 4>, p, G, nrec);
    if (p.lat_dim > 512)
        return wide ? cudaLaunchKernelEx(&cfg, mla_decode_merge_kernel<1, 4, 2>, p, G, nrec)
                    : cudaLaunchKernelEx(&cfg, mla_decode_merge_kernel<2, 1, 2>, p, G, nrec);
    return wide ? cudaLaunchKernelEx(&cfg, mla_decode_merge_kernel<1, 4, 1>, p, G, nrec)
                : cudaLaunchKernelEx(&cfg, mla_decode_merge_kernel<2, 1, 1>, p, G, nrec);
}

template <int NP, bool LSU, int KIND>
struct Variant {
    static constexpr int kThreads = decode_threads<LSU, KIND>();

    // Set the shared-memory attribute (once per device) and return how many
    // clusters of 2 fit on the device at once.
    static int max_clusters() {
        static int done[64] = {0};
        static int clusters[64] = {0};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return -1;
        if (!done[dev]) {
            auto k = mla_decode_kernel<NP, LSU, KIND>;
            if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<NP, LSU>::kSmemBytes) != cudaSuccess)
                return -1;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2, 1, 1);
            cfg.blockDim = dim3(kThreads, 1, 1);
            cfg.dynamicSmemBytes = Cfg<NP, LSU>::kSmemBytes;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess || n <= 0) return -1;
            clusters[dev] = n;
            done[dev] = 1;
        }
        return clusters[dev];
    }

    static cudaError_t launch(const DecodeMaps& maps, const DecodeParams& p, int G, int GY, cudaStream_t stream) {
        cudaLaunchAttribute attr[1];
        cudaLaunchConfig_t cfg = pdl_config(dim3(2 * G, GY), kThreads, Cfg<NP, LSU>::kSmemBytes, stream, attr);
        return cudaLaunchKernelEx(&cfg, mla_decode_kernel<NP, LSU, KIND>, maps, p);
    }
};

template <typename V>
static int pick_clusters(int requested_ctas) {
    const int mx = V::max_clusters();
    if (mx <= 0) return -1;
    if (requested_ctas <= 0) return mx;
    return max(1, requested_ctas / 2);
}

#define MLA_DISPATCH_NP(NPV, EXPR, L, K) \
    (NPV == 16 ? EXPR(16, L, K) : NPV == 32 ? EXPR(32, L, K) : EXPR(64, L, K))
#define MLA_DISPATCH(NPV, EXPR)                                                                            \
    (kind == 1 ? (lsu ? MLA_DISPATCH_NP(NPV, EXPR, true, 1) : MLA_DISPATCH_NP(NPV, EXPR, false, 1)) \
               : (lsu ? MLA_DISPATCH_NP(NPV, EXPR, true, 0) : MLA_DISPATCH_NP(NPV, EXPR, false, 0)))

int decode_clusters(int NP, bool lsu, int kind, int requested_ctas) {
#define MLA_PICK(a, b, c) pick_clusters<Variant<a, b, c>>(requested_ctas)
    return MLA_DISPATCH(NP, MLA_PICK);
#undef MLA_PICK
}

cudaError_t launch_decode(const DecodeMaps& maps, const DecodeParams& p, int NP, bool lsu, int kind, int G, int GY,
                          cudaStream_t stream) {
#define MLA_LAUNCH(a, b, c) Variant<a, b, c>::launch(maps, p, G, GY, stream)
    cudaError_t e = MLA_DISPATCH(NP, MLA_LAUNCH);
#undef MLA_LAUNCH
    if (e != cudaSuccess) return e;
    return launch_decode_merge(p, G, 2 * G * GY, GY, stream);
}

template <int NP, int KB, bool PAIR = false, bool MC = false, int KIND = 0>
struct FoldVariant {
    using C = FoldCfg<NP, KB, PAIR, KIND>;
    static constexpr bool kCluster = PAIR || MC;
    // cluster shape: the latent halves of a row (PAIR) side by side in x, the
    // two row groups (MC) in y
    static void cluster_attr(cudaLaunchAttribute& a) {
        a.id = cudaLaunchAttributeClusterDimension;
        a.val.clusterDim.x = PAIR ? 2 : 1;
        a.val.clusterDim.y = MC ? 2 : 1;
        a.val.clusterDim.z = 1;
    }
    // Set the shared-memory attribute (once per device) and return how many
    // workers (CTAs, or clusters of two) fit on the device at once.
    static int max_workers() {
        static int done[64] = {0};
        static int workers[64] = {0};
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64) return -1;
        if (!done[dev]) {
            auto k = mla_decode_fold_kernel<NP, KB, PAIR, MC, KIND>;
            if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
                return -1;
            if constexpr (kCluster) {
                cudaLaunchConfig_t cfg = {};
                cudaLaunchAttribute attr[1];
                cluster_attr(attr[0]);
                cfg.gridDim = dim3(PAIR ? 2 : 1, MC ? 2 : 1, 1);
                cfg.blockDim = dim3(C::kThreads, 1, 1);
                cfg.dynamicSmemBytes = C::kSmemBytes;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                int n = 0;
                if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess || n <= 0) return -1;
                workers[dev] = n;
            } else {
                int per_sm = 0, sms = 0;
                if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, C::kThreads, C::kSmemBytes) != cudaSuccess ||
                    per_sm <= 0)
                    return -1;
                if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
                    return -1;
                workers[dev] = per_sm * sms;
            }
            done[dev] = 1;
        }
        return workers[dev];
    }

    static cudaError_t launch(const DecodeMaps& maps, const DecodeParams& p, int W, int GY, cudaStream_t stream) {
        cudaLaunchAttribute attr[2];
        cudaLaunchConfig_t cfg = pdl_config(dim3(PAIR ? 2 * W : W, GY), C::kThreads, C::kSmemBytes, stream, attr);
        if constexpr (kCluster) {
            cluster_attr(attr[1]);
            cfg.numAttrs = 2;
        }
        return cudaLaunchKernelEx(&cfg, mla_decode_fold_kernel<NP, KB, PAIR, MC, KIND>, maps, p);
    }
};

// The folded-tile variants: query rows padded to NP, latent width D (K-blocks
// per tile 128 / D; 1792 splits the latent over a CTA pair); at 65 to 128
// query rows of the 576-wide row the two row groups share each tile (MC);
// fp8_ds_mla rows (KINDV 1) at 64 rows.
#define MLA_FOLD(NPV, DV, MCV, KINDV, EXPR)                                                                   \
    (DV == 512 ? (NPV == 16 ? (KINDV ? EXPR(16, 4, false, false, 1) : EXPR(16, 4, false, false, 0))             \
                            : NPV == 32 ? (KINDV ? EXPR(32, 4, false, false, 1) : EXPR(32, 4, false, false, 0)) \
                                        : (MCV ? EXPR(64, 4, false, true, 0)                                   \
                                               : KINDV ? EXPR(64, 4, false, false, 1) : EXPR(64, 4, false, false, 0))) \
               : DV == 256 ? (NPV == 16 ? EXPR(16, 2, false, false, 0) : EXPR(32, 2, false, false, 0))        \
                           : DV == 768 ? EXPR(16, 6, false, false, 0) : EXPR(16, 7, true, false, 0))

bool fold_supported(int NP, int lat_dim, int kind, int GY) {
    if (kind == 1) return lat_dim == 512 && (NP == 16 || NP == 32 || NP == 64) && GY == 1;
    return lat_dim == 512   ? (NP == 16 || NP == 32 || NP == 64)
           : lat_dim == 256 ? (NP == 16 || NP == 32)
                            : ((lat_dim == 768 || lat_dim == 1792) && NP == 16);
}

bool fold_is_pair(int lat_dim) { return lat_dim == 1792; }

bool fold_is_row_pair(int NP, int lat_dim, int GY) { return NP == 64 && lat_dim == 512 && GY == 2; }

int decode_fold_ctas(int NP, int lat_dim, int kind, int GY, int requested_ctas) {
    if (!fold_supported(NP, lat_dim, kind, GY)) return -1;
    const bool mc = kind == 0 && fold_is_row_pair(NP, lat_dim, GY);
#define MLA_FOLD_WORKERS(a, b, c, d, e) FoldVariant<a, b, c, d, e>::max_workers()
    const int mx = MLA_FOLD(NP, lat_dim, mc, kind == 1, MLA_FOLD_WORKERS);
#undef MLA_FOLD_WORKERS
    if (mx <= 0) return -1;
    if (requested_ctas <= 0) return mx;
    if (fold_is_pair(lat_dim)) return requested_ctas >= 4 ? requested_ctas / 2 : 1;
    if (mc) return requested_ctas >= 2 ? requested_ctas / 2 : 1;  // the grid has GY = 2 CTAs per worker
    return requested_ctas;
}

cudaError_t launch_decode_fold(const DecodeMaps& maps, const DecodeParams& p, int NP, int kind, int W, int GY,
                               cudaStream_t stream) {
    if (!fold_supported(NP, p.lat_dim, kind, GY)) return cudaErrorInvalidValue;
    const bool mc = kind == 0 && fold_is_row_pair(NP, p.lat_dim, GY);
#define MLA_FOLD_LAUNCH(a, b, c, d, e) FoldVariant<a, b, c, d, e>::launch(maps, p, W, GY, stream)
    cudaError_t e = MLA_FOLD(NP, p.lat_dim, mc, kind == 1, MLA_FOLD_LAUNCH);
#undef MLA_FOLD_LAUNCH
    if (e != cudaSuccess) return e;
    // status records: one per CTA
    return launch_decode_merge(p, W, (fold_is_pair(p.lat_dim) ? 2 * W : W) * GY, GY, stream);
}

cudaError_t launch_merge_lse(const float* part_o, const float* part_lse, int S, int64_t N, void* out, int out_f32,
                             float* lse, cudaStream_t stream) {
    if (N == 0) return cudaSuccess;
    const int64_t blocks = (N + 7) / 8;
    mla_merge_lse_kernel<<<dim3(static_cast<unsigned>(blocks)), 256, 0, stream>>>(part_o, part_lse, S, N, out,
                                                                                 out_f32, lse);
    return cudaGetLastError();
}

}  // namespace mla

#ifdef MLA_TRACE
extern "C" __attribute__((visibility("default"))) int mla_trace_dump(void* host) {
    return static_cast<int>(cudaMemcpyFromSymbol(host, mla::g_trace, sizeof(mla::g_trace)));
}
extern "C" __attribute__((visibility("default"))) int mla_ttrace_dump(void* ttrace, void* ksm) {
    cudaError_t e = cudaMemcpyFromSymbol(ttrace, mla::g_ttrace, sizeof(mla::g_ttrace));
    if (e != cudaSuccess) return static_cast<int>(e);
    return static_cast<int>(cudaMemcpyFromSymbol(ksm, mla::g_ksm, sizeof(mla::g_ksm)));
}
extern "C" __attribute__((visibility("default"))) int mla_ktrace_dump(void* host) {
    cudaError_t e = cudaMemcpyFromSymbol(host, mla::g_ktrace, sizeof(mla::g_ktrace));
    if (e != cudaSuccess) return static_cast<int>(e);
    return static_cast<int>(cudaMemcpyFromSymbol(static_cast<char*>(host) + sizeof(mla::g_ktrace), mla::g_mtrace,
                                                 sizeof(mla::g_mtrace)));
}
#endif
