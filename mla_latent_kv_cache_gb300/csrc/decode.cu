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
// Work split ("stream-K" over 128-token tiles). The tiles of all requests are
// concatenated and gridDim.x CTAs (one per SM) each take an equal contiguous
// range, so every SM streams the same number of cache bytes whatever the
// request lengths. A CTA walks its range tile by tile; the tiles of one
// request inside a range form a segment. A segment that covers its whole
// request writes the final output; otherwise it writes an fp32 partial
// (out, lse) that a second kernel merges. Rows (query token x head) are
// processed NP at a time (NP = 16, 32 or 64, padded); gridDim.y covers more.
//
// Per tile, all query rows share one read of the cache (the pages' point that
// a verify step must read the latent once per request):
//   S^T[128 tok, NP] = C[128, 576] . Q^T            (UMMA M=128, K=576)
//   P = exp2(S*scale*log2e - m)  (bf16, in smem)
//   O^T[512, NP]    += C[128, 0:512]^T . P^T         (4 UMMAs of M=128, K=128)
// C stays in shared memory in the 128-byte-swizzled layout that serves as the
// K-major A operand of the first product and the MN-major A operand of the
// second. S and O live in tensor memory.
//
// Warp roles (one CTA per SM):
//   warp 0      : TMEM allocation; one lane issues every tcgen05.mma
//   warp 1      : TMA producer (bf16 pools, page_size % 8 == 0)
//   warp 2      : tile-range scan at start
//   warps 4..7  : softmax, P, output epilogue (thread t <-> token t <-> TMEM lane t)
//   warps 8..11 : load/convert producers (fp8 pools or odd page sizes)
//
// Online softmax with a lazily updated maximum: m is raised only when a score
// exceeds it by more than 2^8 (in log2 units), so P <= 256 and rescaling of O
// is rare; l is kept per thread and reduced once per segment.
#include <climits>

#include "launch.cuh"
#include "mla_common.cuh"

namespace mla {

constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.69314718055994530942f;

template <int NP>
struct Cfg {
    static_assert(NP == 16 || NP == 32 || NP == 64, "NP");
    static constexpr int kPairBytes = 2 * 128 * 128;  // two 64-dim chunks of a 128-token tile
    static constexpr int kRopeBytes = 128 * 128;
    static constexpr bool kPInRope = (NP == 64);  // P reuses the tile's rope buffer
    static constexpr int kRL = (NP == 64) ? 4 : 5;
    static constexpr int kRR = (NP == 16) ? 2 : 1;
    static constexpr int kQBytes = 9 * NP * 128;
    static constexpr int kPBytes = kPInRope ? 0 : 128 * NP * 2;
    static constexpr int kOffRope = kRL * kPairBytes;
    static constexpr int kOffQ = kOffRope + kRR * kRopeBytes;
    static constexpr int kOffP = kOffQ + kQBytes;
    static constexpr int kOffCtrl = kOffP + kPBytes;
    static constexpr int kSmemBytes = kOffCtrl + 4096 + 1024;  // + alignment slack
    static constexpr int kTmemCols = (5 * NP <= 128) ? 128 : (5 * NP <= 256) ? 256 : 512;
    static constexpr int kColS = 4 * NP;
    // P operand: MN-major rows of NP bf16, swizzle span = row width
    static constexpr uint32_t kPSwizzle = NP == 16 ? kSw32 : NP == 32 ? kSw64 : kSw128;
    static_assert(kSmemBytes <= 232448, "shared memory");
};

struct Ctrl {
    uint64_t pair_full[5], pair_empty[5];
    uint64_t rope_full[2], rope_empty[2];
    uint64_t s_full, p_full, o_done, q_full;
    uint32_t tmem_base;
    int abort;
    int t_begin, t_end, b0, j0;
    int colvis[64];       // query row -> how many trailing tokens it may not see
    float m[64];          // running max per row (log2 units)
    float alpha[64];
    float red[4][64];
};

// Column c of this row group may see token `tok` of a request of length T iff
// tok + colvis[c] < T; padded columns never see anything.
__device__ __forceinline__ int swz_p(int row, uint32_t mode) {
    return mode == kSw128 ? (row & 7) : mode == kSw64 ? ((row >> 1) & 3) : ((row >> 2) & 1);
}

struct TileIt {
    int b, j, tiles, T;
    __device__ __forceinline__ void init(const int32_t* sl, int b0, int j0) {
        b = b0;
        j = j0;
        T = max(__ldg(sl + b), 0);
        tiles = (T + kTile - 1) / kTile;
    }
    __device__ __forceinline__ void next(const int32_t* sl, int B) {
        if (++j >= tiles) {
            j = 0;
            do {
                ++b;
                if (b >= B) { T = 0; tiles = 1; break; }
                T = max(__ldg(sl + b), 0);
                tiles = (T + kTile - 1) / kTile;
            } while (tiles == 0);
        }
    }
};

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
    if constexpr (NP == 16) tmem_ld_x16(taddr, r);
    else if constexpr (NP == 32) tmem_ld_x32(taddr, r);
    else tmem_ld_x64(taddr, r);
}
template <int NP>
__device__ __forceinline__ void tmem_st_np(uint32_t taddr, const uint32_t (&r)[NP]) {
    if constexpr (NP == 16) tmem_st_x16(taddr, r);
    else if constexpr (NP == 32) tmem_st_x32(taddr, r);
    else tmem_st_x64(taddr, r);
}

__device__ __forceinline__ void fail(const DecodeParams& p, Ctrl* ctrl, int code) {
    atomicOr(p.status, code);
    ctrl->abort = 1;
}

// Every softmax thread waits, then the 128 threads agree on the outcome, so a
// timeout seen by some of them cannot strand the rest at a named barrier.
__device__ __forceinline__ bool group_wait(uint64_t* bar, uint32_t parity, const DecodeParams& p, Ctrl* ctrl) {
    const bool ok = mbar_wait(bar, parity, &ctrl->abort);
    const bool all = named_bar_and(3, 128, ok ? 1 : 0) != 0;
    if (!ok) fail(p, ctrl, kErrWaitTimeout);
    return all;
}

// Load the NP query rows of request b (row group gy) into the K-major,
// 128-byte-swizzled B operand: chunk k (64 dims) at k*NP*128, row n at n*128.
template <int NP>
__device__ void load_q(const DecodeParams& p, int b, int gy, uint8_t* qs, int tid) {
    for (int q = tid; q < NP * 72; q += 128) {
        const int n = q / 72, u = q - n * 72;
        const int r = gy * 64 + n;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r < p.HQ) {
            const int64_t row = static_cast<int64_t>(b) * p.HQ + r;
            v = (u < 64) ? __ldg(reinterpret_cast<const uint4*>(p.q_lat + row * kD) + u)
                         : __ldg(reinterpret_cast<const uint4*>(p.q_pe + row * kP) + (u - 64));
        }
        const int chunk = u >> 3, uu = u & 7;
        *reinterpret_cast<uint4*>(qs + chunk * NP * 128 + n * 128 + ((uu ^ (n & 7)) << 4)) = v;
    }
}

// 64-bit slot of token `tok` of the request whose block-table row is `btr`.
__device__ __forceinline__ int64_t token_slot(const DecodeParams& p, const int32_t* btr, int tok, bool& bad) {
    const int64_t page = __ldg(btr + tok / p.page_size);
    const int64_t ps = p.page_size;
    if (page < 0 || (page + 1) * ps > p.num_slots) {
        bad = true;
        return tok % p.page_size;  // page 0: in bounds, flagged
    }
    return page * ps + tok % p.page_size;
}

// e4m3 x16 (one uint4) times scale -> 16 bf16 (two uint4).
__device__ __forceinline__ void dequant16(uint4 codes, float scale, uint4& lo, uint4& hi) {
    const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __half2_raw h01 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] & 0xFFFFu), __NV_E4M3);
        const __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[i] >> 16), __NV_E4M3);
        const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
        const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
        o[2 * i] = pack_bf16x2(f01.x * scale, f01.y * scale);
        o[2 * i + 1] = pack_bf16x2(f23.x * scale, f23.y * scale);
    }
    lo = make_uint4(o[0], o[1], o[2], o[3]);
    hi = make_uint4(o[4], o[5], o[6], o[7]);
}

template <int NP, bool LSU, int KIND>
__global__ void __launch_bounds__(LSU ? 384 : 256, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tmap, const DecodeParams p) {
    using C = Cfg<NP>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* pair_ring = smem;
    uint8_t* rope_ring = smem + C::kOffRope;
    uint8_t* qs = smem + C::kOffQ;
    uint8_t* pbuf = smem + C::kOffP;
    Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + C::kOffCtrl);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = blockIdx.x, G = gridDim.x, gy = blockIdx.y;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kRL; ++i) { mbar_init(&ctrl->pair_full[i], 1); mbar_init(&ctrl->pair_empty[i], 1); }
        for (int i = 0; i < C::kRR; ++i) { mbar_init(&ctrl->rope_full[i], 1); mbar_init(&ctrl->rope_empty[i], 1); }
        mbar_init(&ctrl->s_full, 1);
        mbar_init(&ctrl->p_full, 1);
        mbar_init(&ctrl->o_done, 1);
        mbar_init(&ctrl->q_full, 1);
        ctrl->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&ctrl->tmem_base, C::kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    if (!LSU && warp == 1 && lane == 0) prefetch_tensormap(&tmap);
    if (warp == 2) {
        // tiles per request, their total, and where this CTA's range starts
        long long total = 0;
        for (int base = 0; base < p.B; base += 32) {
            const int b = base + lane;
            const int tl = b < p.B ? (max(__ldg(p.seq_lens + b), 0) + kTile - 1) / kTile : 0;
            int s = tl;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            total += s;
        }
        const int tb = static_cast<int>(static_cast<long long>(g) * total / G);
        const int te = static_cast<int>(static_cast<long long>(g + 1) * total / G);
        int b0 = 0, j0 = 0;
        long long acc = 0;
        for (int base = 0; base < p.B && tb < te; base += 32) {
            const int b = base + lane;
            const int tl = b < p.B ? (max(__ldg(p.seq_lens + b), 0) + kTile - 1) / kTile : 0;
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
        if (lane == 0) {
            ctrl->t_begin = tb;
            ctrl->t_end = te;
            ctrl->b0 = b0;
            ctrl->j0 = j0;
        }
    }
    if (threadIdx.x >= 128 && threadIdx.x < 128 + 64) {
        const int c = threadIdx.x - 128;
        const int r = gy * 64 + c;
        ctrl->colvis[c] = (r < p.HQ) ? (p.Qt - 1 - r / p.Hq) : (INT_MAX / 2);
        ctrl->m[c] = -INFINITY;
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    const int ntiles = ctrl->t_end - ctrl->t_begin;

    if (ntiles > 0) {
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------------ MMA issuer
            TileIt it;
            it.init(p.seq_lens, ctrl->b0, ctrl->j0);
            const uint32_t idS = idesc_bf16(128, NP, false, false);
            const uint32_t idPV = idesc_bf16(128, NP, true, true);
            const uint32_t q_addr = smem_u32(qs);
            const uint32_t tS = tmem + C::kColS;
            int seg = 0;
            for (int i = 0; i < ntiles; ++i) {
                const bool new_seg = (i == 0) || (it.j == 0);
                if (new_seg) {
                    if (!mbar_wait(&ctrl->q_full, seg & 1, &ctrl->abort)) { fail(p, ctrl, kErrWaitTimeout); break; }
                    ++seg;
                }
                bool ok = true;
                for (int pp = 0; pp < 4 && ok; ++pp) {
                    const int u = 4 * i + pp, slot = u % C::kRL;
                    if (!mbar_wait(&ctrl->pair_full[slot], (u / C::kRL) & 1, &ctrl->abort)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t base = smem_u32(pair_ring + slot * C::kPairBytes);
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t a = smem_desc(base + c * 16384 + kk * 32, 16, 1024, kSw128);
                            const uint64_t bq = smem_desc(q_addr + (2 * pp + c) * NP * 128 + kk * 32, 16, 1024, kSw128);
                            umma_bf16(tS, a, bq, idS, (pp | c | kk) != 0);
                        }
                }
                const int rr = i % C::kRR;
                if (ok && !mbar_wait(&ctrl->rope_full[rr], (i / C::kRR) & 1, &ctrl->abort)) ok = false;
                if (!ok) { fail(p, ctrl, kErrWaitTimeout); break; }
                tc_fence_after();
                const uint32_t rbase = smem_u32(rope_ring + rr * C::kRopeBytes);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t a = smem_desc(rbase + kk * 32, 16, 1024, kSw128);
                    const uint64_t bq = smem_desc(q_addr + 8 * NP * 128 + kk * 32, 16, 1024, kSw128);
                    umma_bf16(tS, a, bq, idS, 1u);
                }
                umma_commit(&ctrl->s_full);
                if (!C::kPInRope) umma_commit(&ctrl->rope_empty[rr]);

                if (!mbar_wait(&ctrl->p_full, i & 1, &ctrl->abort)) { fail(p, ctrl, kErrWaitTimeout); break; }
                tc_fence_after();
                const uint32_t paddr = C::kPInRope ? rbase : smem_u32(pbuf);
                constexpr uint32_t p_sbo = 8 * NP * 2;
#pragma unroll
                for (int mt = 0; mt < 4; ++mt) {
                    const int slot = (4 * i + mt) % C::kRL;
                    const uint32_t base = smem_u32(pair_ring + slot * C::kPairBytes);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t a = smem_desc(base + kk * 2048, 16384, 1024, kSw128);
                        const uint64_t bp = smem_desc(paddr + kk * 16 * NP * 2, p_sbo, p_sbo, C::kPSwizzle);
                        umma_bf16(tmem + mt * NP, a, bp, idPV, (new_seg && kk == 0) ? 0u : 1u);
                    }
                    umma_commit(&ctrl->pair_empty[slot]);
                }
                if (C::kPInRope) umma_commit(&ctrl->rope_empty[rr]);
                umma_commit(&ctrl->o_done);
                it.next(p.seq_lens, p.B);
            }
        } else if (!LSU && warp == 1 && lane == 0) {
            // ------------------------------------------------- TMA producer
            TileIt it;
            it.init(p.seq_lens, ctrl->b0, ctrl->j0);
            const uint64_t pol = l2_policy_evict_first();
            const int BR = p.run_rows;
            bool bad = false, ok = true;
            for (int i = 0; i < ntiles && ok; ++i) {
                const int valid = min(kTile, it.T - it.j * kTile);
                const int nruns = (valid + BR - 1) / BR;
                const int32_t* btr = p.block_table + static_cast<int64_t>(it.b) * p.bt_stride;
                int ys[16];
                for (int r = 0; r < nruns; ++r)
                    ys[r] = static_cast<int>(token_slot(p, btr, it.j * kTile + r * BR, bad));
                const uint32_t bytes = static_cast<uint32_t>(nruns * BR * 128);
                for (int pp = 0; pp < 4; ++pp) {
                    const int u = 4 * i + pp, slot = u % C::kRL;
                    if (u >= C::kRL && !mbar_wait(&ctrl->pair_empty[slot], ((u / C::kRL) - 1) & 1, &ctrl->abort)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&ctrl->pair_full[slot], 2 * bytes);
                    uint8_t* dst = pair_ring + slot * C::kPairBytes;
                    for (int r = 0; r < nruns; ++r)
#pragma unroll
                        for (int c = 0; c < 2; ++c)
                            tma_load_2d(dst + c * 16384 + r * BR * 128, &tmap, &ctrl->pair_full[slot],
                                        128 * pp + 64 * c, ys[r], pol);
                }
                if (!ok) break;
                const int rr = i % C::kRR;
                if (i >= C::kRR && !mbar_wait(&ctrl->rope_empty[rr], ((i / C::kRR) - 1) & 1, &ctrl->abort)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&ctrl->rope_full[rr], bytes);
                for (int r = 0; r < nruns; ++r)
                    tma_load_2d(rope_ring + rr * C::kRopeBytes + r * BR * 128, &tmap, &ctrl->rope_full[rr], 512,
                                ys[r], pol);
                it.next(p.seq_lens, p.B);
            }
            if (!ok) fail(p, ctrl, kErrWaitTimeout);
            if (bad) atomicOr(p.status, kErrBadBlock);
        } else if (LSU && warp >= 8) {
            // ------------------------------------- load/convert producers
            const int pw = warp - 8;
            TileIt it;
            it.init(p.seq_lens, ctrl->b0, ctrl->j0);
            int ti = 0;
            bool bad = false, ok = true;
            const int rb = KIND == 0 ? kRowBf16 : kRowFp8;
            for (int f = pw; f < ntiles * 5 && ok; f += 4) {
                const int i = f / 5, k = f - 5 * (f / 5);
                while (ti < i) { it.next(p.seq_lens, p.B); ++ti; }
                const int valid = min(kTile, it.T - it.j * kTile);
                const int32_t* btr = p.block_table + static_cast<int64_t>(it.b) * p.bt_stride;
                uint64_t* full;
                uint8_t* dst;
                if (k < 4) {
                    const int u = 4 * i + k, slot = u % C::kRL;
                    if (u >= C::kRL &&
                        !__all_sync(0xffffffffu, mbar_wait(&ctrl->pair_empty[slot], ((u / C::kRL) - 1) & 1, &ctrl->abort))) {
                        ok = false;
                        break;
                    }
                    full = &ctrl->pair_full[slot];
                    dst = pair_ring + slot * C::kPairBytes;
                    if (KIND == 0) {
                        // 16 units of 16 B per token: dims [128k, 128k+128)
                        for (int q0 = 0; q0 < valid * 16; q0 += 128) {
                            uint4 v[4];
                            int tl[4], uu[4];
#pragma unroll
                            for (int s = 0; s < 4; ++s) {
                                const int q = q0 + s * 32 + lane;
                                tl[s] = q >> 4;
                                uu[s] = q & 15;
                                if (tl[s] < valid) {
                                    const int64_t slot64 = token_slot(p, btr, it.j * kTile + tl[s], bad);
                                    v[s] = __ldg(reinterpret_cast<const uint4*>(p.cache + slot64 * rb + k * 256) + uu[s]);
                                }
                            }
#pragma unroll
                            for (int s = 0; s < 4; ++s)
                                if (tl[s] < valid) {
                                    const int c = uu[s] >> 3, un = uu[s] & 7;
                                    *reinterpret_cast<uint4*>(dst + c * 16384 + tl[s] * 128 + ((un ^ (tl[s] & 7)) << 4)) = v[s];
                                }
                        }
                    } else {
                        // 8 units of 16 codes per token, block scale k
                        for (int q0 = 0; q0 < valid * 8; q0 += 128) {
                            uint4 v[4];
                            float sc[4];
                            int tl[4], uu[4];
#pragma unroll
                            for (int s = 0; s < 4; ++s) {
                                const int q = q0 + s * 32 + lane;
                                tl[s] = q >> 3;
                                uu[s] = q & 7;
                                if (tl[s] < valid) {
                                    const int64_t slot64 = token_slot(p, btr, it.j * kTile + tl[s], bad);
                                    const uint8_t* row = p.cache + slot64 * rb;
                                    v[s] = __ldg(reinterpret_cast<const uint4*>(row + k * 128) + uu[s]);
                                    sc[s] = __ldg(reinterpret_cast<const float*>(row + 512) + k);
                                }
                            }
#pragma unroll
                            for (int s = 0; s < 4; ++s)
                                if (tl[s] < valid) {
                                    uint4 lo, hi;
                                    dequant16(v[s], sc[s], lo, hi);
                                    const int c = uu[s] >> 2, un = (uu[s] & 3) * 2;
                                    uint8_t* rowp = dst + c * 16384 + tl[s] * 128;
                                    *reinterpret_cast<uint4*>(rowp + ((un ^ (tl[s] & 7)) << 4)) = lo;
                                    *reinterpret_cast<uint4*>(rowp + (((un + 1) ^ (tl[s] & 7)) << 4)) = hi;
                                }
                        }
                    }
                } else {
                    const int rr = i % C::kRR;
                    if (i >= C::kRR &&
                        !__all_sync(0xffffffffu, mbar_wait(&ctrl->rope_empty[rr], ((i / C::kRR) - 1) & 1, &ctrl->abort))) {
                        ok = false;
                        break;
                    }
                    full = &ctrl->rope_full[rr];
                    dst = rope_ring + rr * C::kRopeBytes;
                    const int roff = KIND == 0 ? 1024 : 528;
                    for (int q0 = 0; q0 < valid * 8; q0 += 128) {
                        uint4 v[4];
                        int tl[4], uu[4];
#pragma unroll
                        for (int s = 0; s < 4; ++s) {
                            const int q = q0 + s * 32 + lane;
                            tl[s] = q >> 3;
                            uu[s] = q & 7;
                            if (tl[s] < valid) {
                                const int64_t slot64 = token_slot(p, btr, it.j * kTile + tl[s], bad);
                                v[s] = __ldg(reinterpret_cast<const uint4*>(p.cache + slot64 * rb + roff) + uu[s]);
                            }
                        }
#pragma unroll
                        for (int s = 0; s < 4; ++s)
                            if (tl[s] < valid)
                                *reinterpret_cast<uint4*>(dst + tl[s] * 128 + ((uu[s] ^ (tl[s] & 7)) << 4)) = v[s];
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(full);
            }
            if (!ok && lane == 0) fail(p, ctrl, kErrWaitTimeout);
            if (bad) atomicOr(p.status, kErrBadBlock);
        } else if (warp >= 4 && warp < 8) {
            // ------------------------------------------ softmax + epilogue
            const int st = threadIdx.x - 128;  // token row of the tile / TMEM lane
            const int sw = warp - 4;
            const uint32_t lane_base = static_cast<uint32_t>(sw * 32) << 16;
            const int HQg = min(64, p.HQ - gy * 64);
            TileIt it;
            it.init(p.seq_lens, ctrl->b0, ctrl->j0);
            float l[NP];
#pragma unroll
            for (int c = 0; c < NP; ++c) l[c] = 0.f;
            int seg_start_j = it.j;
            bool seg_has_pv = false;
            load_q<NP>(p, it.b, gy, qs, st);
            fence_proxy_async_smem();
            named_bar_sync(1, 128);
            if (st == 0) mbar_arrive(&ctrl->q_full);
            for (int i = 0; i < ntiles; ++i) {
                const int b = it.b, j = it.j, T = it.T;
                const bool last_of_seg = (j == it.tiles - 1) || (i == ntiles - 1);
                if (!group_wait(&ctrl->s_full, i & 1, p, ctrl)) break;
                tc_fence_after();
                __syncwarp();
                uint32_t sr[NP];
                tmem_ld_np<NP>(tmem + lane_base + C::kColS, sr);
                if (last_of_seg && i + 1 < ntiles) {
                    // S of this tile is complete, so Q may be replaced by the next request's
                    TileIt nx = it;
                    nx.next(p.seq_lens, p.B);
                    load_q<NP>(p, nx.b, gy, qs, st);
                    fence_proxy_async_smem();
                    named_bar_sync(1, 128);
                    if (st == 0) mbar_arrive(&ctrl->q_full);
                }
                const int tok = j * kTile + st;
                const bool all_vis = (j * kTile + kTile + p.Qt - 1) <= T;
                float x[NP];
                int need = 0;
#pragma unroll
                for (int c = 0; c < NP; ++c) {
                    const bool v = all_vis ? (c < HQg) : (tok + ctrl->colvis[c] < T);
                    x[c] = v ? __uint_as_float(sr[c]) * p.scale_log2 : -INFINITY;
                    need |= (x[c] > ctrl->m[c] + kRescaleThreshold) ? 1 : 0;
                }
                need = named_bar_or(2, 128, need);
                if (need) {
#pragma unroll
                    for (int c = 0; c < NP; ++c) {
                        const float v = warp_max(x[c]);
                        if (lane == 0) ctrl->red[sw][c] = v;
                    }
                    named_bar_sync(1, 128);
                    if (st < NP) {
                        const float mt = fmaxf(fmaxf(ctrl->red[0][st], ctrl->red[1][st]),
                                               fmaxf(ctrl->red[2][st], ctrl->red[3][st]));
                        const float mo = ctrl->m[st];
                        const float mn = fmaxf(mo, mt);
                        ctrl->alpha[st] = (mo == -INFINITY) ? 0.f : ex2(mo - mn);
                        ctrl->m[st] = mn;
                    }
                    named_bar_sync(1, 128);
#pragma unroll
                    for (int c = 0; c < NP; ++c) l[c] *= ctrl->alpha[c];
                    if (seg_has_pv) {
                        // O holds earlier tiles of this segment: wait for the last PV, rescale
                        if (!group_wait(&ctrl->o_done, (i - 1) & 1, p, ctrl)) break;
                        tc_fence_after();
                        __syncwarp();
#pragma unroll 1
                        for (int mt = 0; mt < 4; ++mt) {
                            uint32_t o[NP];
                            tmem_ld_np<NP>(tmem + lane_base + mt * NP, o);
#pragma unroll
                            for (int c = 0; c < NP; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * ctrl->alpha[c]);
                            tmem_st_np<NP>(tmem + lane_base + mt * NP, o);
                        }
                        tmem_wait_st();
                    }
                }
#pragma unroll
                for (int c = 0; c < NP; ++c) {
                    const float pc = (x[c] == -INFINITY) ? 0.f : ex2(x[c] - ctrl->m[c]);
                    l[c] += pc;
                    x[c] = pc;
                }
                // P row `st`: NP bf16, MN-major, swizzled like the MMA reads it
                uint8_t* prow = (C::kPInRope ? rope_ring + (i % C::kRR) * C::kRopeBytes : pbuf) + st * NP * 2;
                const int sz = swz_p(st, C::kPSwizzle);
#pragma unroll
                for (int u = 0; u < NP / 8; ++u) {
                    const uint4 v = make_uint4(pack_bf16x2(x[8 * u + 0], x[8 * u + 1]), pack_bf16x2(x[8 * u + 2], x[8 * u + 3]),
                                               pack_bf16x2(x[8 * u + 4], x[8 * u + 5]), pack_bf16x2(x[8 * u + 6], x[8 * u + 7]));
                    *reinterpret_cast<uint4*>(prow + ((u ^ sz) << 4)) = v;
                }
                if (tok >= T) {
                    // rows past the request hold stale data (possibly NaN); P is 0
                    // there, but 0 * NaN would still poison O, so clear them
                    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                    for (int pp = 0; pp < 4; ++pp) {
                        uint8_t* ps = pair_ring + ((4 * i + pp) % C::kRL) * C::kPairBytes + st * 128;
#pragma unroll
                        for (int c = 0; c < 2; ++c)
#pragma unroll
                            for (int u = 0; u < 8; ++u) *reinterpret_cast<uint4*>(ps + c * 16384 + u * 16) = z;
                    }
                }
                fence_proxy_async_smem();
                tc_fence_before();
                named_bar_sync(1, 128);
                if (st == 0) mbar_arrive(&ctrl->p_full);
                seg_has_pv = true;

                if (last_of_seg) {
                    // ------------------------------------------- epilogue
                    if (!group_wait(&ctrl->o_done, i & 1, p, ctrl)) break;
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < NP; ++c) {
                        const float v = warp_sum(l[c]);
                        if (lane == 0) ctrl->red[sw][c] = v;
                    }
                    named_bar_sync(1, 128);
                    const bool final_seg = (seg_start_j == 0) && (j == it.tiles - 1);
                    __syncwarp();
                    const int64_t pslot = static_cast<int64_t>(gy) * p.SPG + g + b;
#pragma unroll 1
                    for (int mt = 0; mt < 4; ++mt) {
                        uint32_t o[NP];
                        tmem_ld_np<NP>(tmem + lane_base + mt * NP, o);
                        const int d = mt * 128 + st;
#pragma unroll
                        for (int c = 0; c < NP; ++c) {
                            if (c >= HQg) break;
                            const float lt = ctrl->red[0][c] + ctrl->red[1][c] + ctrl->red[2][c] + ctrl->red[3][c];
                            const float v = lt > 0.f ? __uint_as_float(o[c]) / lt : 0.f;
                            if (final_seg) {
                                const int64_t idx = (static_cast<int64_t>(b) * p.HQ + gy * 64 + c) * kD + d;
                                if (p.out_f32) static_cast<float*>(p.out)[idx] = v;
                                else static_cast<__nv_bfloat16*>(p.out)[idx] = __float2bfloat16_rn(v);
                            } else {
                                p.part_o[(pslot * 64 + c) * kD + d] = v;
                            }
                        }
                    }
                    if (st < HQg) {
                        const float lt = ctrl->red[0][st] + ctrl->red[1][st] + ctrl->red[2][st] + ctrl->red[3][st];
                        const float lv = lt > 0.f ? (ctrl->m[st] + log2f(lt)) * kLn2 : -INFINITY;
                        if (final_seg) p.lse[static_cast<int64_t>(b) * p.HQ + gy * 64 + st] = lv;
                        else p.part_lse[pslot * 64 + st] = lv;
                    }
                    tc_fence_before();
                    named_bar_sync(1, 128);
                    if (st < NP) ctrl->m[st] = -INFINITY;
#pragma unroll
                    for (int c = 0; c < NP; ++c) l[c] = 0.f;
                    named_bar_sync(1, 128);
                    seg_has_pv = false;
                    seg_start_j = 0;
                }
                it.next(p.seq_lens, p.B);
            }
        }
    }
    __syncthreads();
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
// CTA g of G got tiles [g*tot/G, (g+1)*tot/G); with more CTAs than tiles some
// ranges are empty and wrote no partial. tot == 0 means "all partials live".
__device__ __forceinline__ bool seg_live(long long tot, int G, long long g) {
    return tot == 0 || (g * tot / G) < ((g + 1) * tot / G);
}

__device__ __forceinline__ void merge_row(const float* po, int64_t o_stride, const float* pl, int64_t l_stride,
                                          int nseg, void* out, int out_f32, float* lse_out, int lane,
                                          long long tot = 0, int G = 1, long long g0 = 0) {
    float mx = -INFINITY;
    for (int s = lane; s < nseg; s += 32)
        if (seg_live(tot, G, g0 + s)) mx = fmaxf(mx, pl[s * l_stride]);
    mx = warp_max(mx);
    float4 acc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    float L = -INFINITY;
    if (mx != -INFINITY) {
        float ws = 0.f;
        for (int s = lane; s < nseg; s += 32) {
            if (!seg_live(tot, G, g0 + s)) continue;
            const float v = pl[s * l_stride];
            if (v != -INFINITY) ws += expf(v - mx);
        }
        ws = warp_sum(ws);
        L = mx + logf(ws);
        for (int s = 0; s < nseg; ++s) {
            if (!seg_live(tot, G, g0 + s)) continue;
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

// Per request b (blockIdx.x) and row group (blockIdx.y): merge the partials
// of a request cut across CTAs, and write (0, -inf) for empty requests.
__global__ void __launch_bounds__(256) mla_decode_merge_kernel(const DecodeParams p, int G) {
    const int b = blockIdx.x, gy = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    __shared__ long long red_pre[8], red_tot[8];
    long long pre = 0, tot = 0;
    for (int i = tid; i < p.B; i += 256) {
        const long long tl = (max(__ldg(p.seq_lens + i), 0) + kTile - 1) / kTile;
        tot += tl;
        if (i < b) pre += tl;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        pre += __shfl_xor_sync(0xffffffffu, pre, o);
        tot += __shfl_xor_sync(0xffffffffu, tot, o);
    }
    if (lane == 0) { red_pre[warp] = pre; red_tot[warp] = tot; }
    __syncthreads();
    pre = 0;
    tot = 0;
    for (int w = 0; w < 8; ++w) { pre += red_pre[w]; tot += red_tot[w]; }
    const int tiles_b = (max(__ldg(p.seq_lens + b), 0) + kTile - 1) / kTile;
    const int HQg = min(64, p.HQ - gy * 64);
    if (tiles_b == 0) {
        for (int n = warp; n < HQg; n += 8) {
            const int64_t row = static_cast<int64_t>(b) * p.HQ + gy * 64 + n;
            merge_row(nullptr, 0, nullptr, 0, 0, static_cast<uint8_t*>(p.out) + row * kD * (p.out_f32 ? 4 : 2),
                      p.out_f32, p.lse + row, lane);
        }
        return;
    }
    // CTA holding tile t: the largest g with floor(g * tot / G) <= t
    const long long g0 = ((pre + 1) * G - 1) / tot;
    const long long g1 = ((pre + tiles_b) * G - 1) / tot;
    if (g0 == g1) return;  // one CTA held the whole request and wrote the output
    const int nseg = static_cast<int>(g1 - g0 + 1);
    const int64_t slot0 = static_cast<int64_t>(gy) * p.SPG + g0 + b;
    for (int n = warp; n < HQg; n += 8) {
        const int64_t row = static_cast<int64_t>(b) * p.HQ + gy * 64 + n;
        merge_row(p.part_o + (slot0 * 64 + n) * kD, 64 * kD, p.part_lse + slot0 * 64 + n, 64, nseg,
                  static_cast<uint8_t*>(p.out) + row * kD * (p.out_f32 ? 4 : 2), p.out_f32, p.lse + row, lane,
                  tot, G, g0);
    }
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

template <int NP, bool LSU, int KIND>
static cudaError_t launch_variant(const CUtensorMap& tmap, const DecodeParams& p, int G, int GY, cudaStream_t stream) {
    using C = Cfg<NP>;
    auto kern = mla_decode_kernel<NP, LSU, KIND>;
    static int attr_done[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_done[dev] = 1;
    }
    kern<<<dim3(G, GY), LSU ? 384 : 256, C::kSmemBytes, stream>>>(tmap, p);
    return cudaGetLastError();
}

cudaError_t launch_decode(const CUtensorMap& tmap, const DecodeParams& p, int NP, bool lsu, int kind, int G, int GY,
                          cudaStream_t stream) {
    cudaError_t e;
    if (kind == 1) {
        e = NP == 16 ? launch_variant<16, true, 1>(tmap, p, G, GY, stream)
          : NP == 32 ? launch_variant<32, true, 1>(tmap, p, G, GY, stream)
                     : launch_variant<64, true, 1>(tmap, p, G, GY, stream);
    } else if (lsu) {
        e = NP == 16 ? launch_variant<16, true, 0>(tmap, p, G, GY, stream)
          : NP == 32 ? launch_variant<32, true, 0>(tmap, p, G, GY, stream)
                     : launch_variant<64, true, 0>(tmap, p, G, GY, stream);
    } else {
        e = NP == 16 ? launch_variant<16, false, 0>(tmap, p, G, GY, stream)
          : NP == 32 ? launch_variant<32, false, 0>(tmap, p, G, GY, stream)
                     : launch_variant<64, false, 0>(tmap, p, G, GY, stream);
    }
    if (e != cudaSuccess) return e;
    mla_decode_merge_kernel<<<dim3(p.B, GY), 256, 0, stream>>>(p, G);
    return cudaGetLastError();
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
