// C ABI entry points (declared in include/mla.h): host-side validation,
// launch planning and TMA descriptor set-up. No entry point allocates memory
// or synchronises.
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <atomic>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "mla.h"
#include "launch.cuh"
#include "mla_common.cuh"

namespace {

constexpr size_t kWsHeader = 256;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DevInfo {
    int sms = -1;
    int major = 0, minor = 0;
};

DevInfo dev_info(int dev) {
    static std::mutex mu;
    static DevInfo cache[64];
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 0 || dev >= 64) return DevInfo{};
    if (cache[dev].sms < 0) {
        DevInfo d;
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DevInfo{};
        cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
        cache[dev] = d;
    }
    return cache[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

int gcd_int(int a, int b) {
    while (b) {
        const int t = a % b;
        a = b;
        b = t;
    }
    return a;
}

int rows_padded(int rows) { return rows <= 16 ? 16 : rows <= 32 ? 32 : 64; }

// Workspace for a grid of `ctas` CTAs: [header 256 B][per-CTA status
// records][partial LSEs][partial outputs], each part 256-byte aligned, with
// ctas + B partial slots per row group (a worker, a CTA or a cluster of two,
// cuts at most one request that another worker continues).
struct WsLayout {
    size_t rec_off, lse_off, o_off, total;
};

WsLayout decode_ws_layout(int B, int HQ, int ctas, int D = 512) {
    const size_t GY = (static_cast<size_t>(HQ) + 63) / 64;
    const size_t slots = GY * static_cast<size_t>(ctas + B) * 64;
    const size_t rec_bytes = (static_cast<size_t>(ctas) * GY * mla::kStatusRecWords * sizeof(int) + 255) / 256 * 256;
    const size_t lse_bytes = (slots * sizeof(float) + 255) / 256 * 256;
    WsLayout l;
    l.rec_off = kWsHeader;
    l.lse_off = l.rec_off + rec_bytes;
    l.o_off = l.lse_off + lse_bytes;
    l.total = l.o_off + slots * static_cast<size_t>(D) * sizeof(float);
    return l;
}

// CTAs the workspace is sized for: num_ctas, or one per SM when 0; at least
// one cluster of two.
int ws_ctas(int num_ctas, int sms) { return num_ctas > 0 ? (num_ctas < 2 ? 2 : num_ctas) : (sms < 2 ? 2 : sms); }

size_t decode_ws_bytes(int B, int HQ, int ctas, int D = 512) { return decode_ws_layout(B, HQ, ctas, D).total; }

// Set by mla_test_hold_next_decode (1) or mla_test_slow_pv_next_decode (2),
// consumed by the next mla_decode.
std::atomic<int> g_test_hold{0};

// Workspace of mla_decode_static_scratch: one array per device, placed when
// this library's device code is loaded, for callers that cannot allocate.
static __device__ __align__(256) unsigned char g_decode_scratch[MLA_STATIC_SCRATCH_BYTES];

// Its address on the current device, looked up once per device.
void* decode_scratch_ptr() {
    static std::mutex mu;
    static void* ptr[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess) return nullptr;
        ptr[dev] = p;
    }
    return ptr[dev];
}

}  // namespace

extern "C" {

int mla_row_bytes(int cache_kind) {
    return cache_kind == MLA_CACHE_BF16_576 ? mla::kRowBf16 : cache_kind == MLA_CACHE_FP8_DS_MLA_656 ? mla::kRowFp8 : 0;
}

const char* mla_status_string(int status) {
    switch (status) {
        case MLA_OK: return "ok";
        case MLA_ERR_INVALID_ARG: return "invalid argument";
        case MLA_ERR_UNSUPPORTED: return "unsupported configuration or device";
        case MLA_ERR_WORKSPACE: return "workspace too small";
        case MLA_ERR_CUDA: return "CUDA error";
        case MLA_ERR_SCRATCH_LIMIT: return "call needs more than the static decode scratch holds";
        default: return "unknown status";
    }
}

int mla_num_sms(void) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    return dev_info(dev).sms;
}

int mla_cache_write(const void* latent, int64_t latent_stride, const void* k_pe, int64_t k_pe_stride,
                    const int64_t* slot_mapping, int64_t num_tokens, void* cache, int64_t num_slots, int cache_kind,
                    int32_t* status, void* stream) {
    if (num_tokens < 0 || num_slots < 0) return MLA_ERR_INVALID_ARG;
    if (cache_kind != MLA_CACHE_BF16_576 && cache_kind != MLA_CACHE_FP8_DS_MLA_656) return MLA_ERR_INVALID_ARG;
    if (num_tokens == 0) return MLA_OK;
    if (!latent || !k_pe || !slot_mapping || !cache) return MLA_ERR_INVALID_ARG;
    if (!aligned16(latent) || !aligned16(k_pe) || !aligned16(cache)) return MLA_ERR_INVALID_ARG;
    if (latent_stride < mla::kD || latent_stride % 8 || k_pe_stride < mla::kP || k_pe_stride % 8)
        return MLA_ERR_INVALID_ARG;
    if (status && (reinterpret_cast<uintptr_t>(status) & 3u)) return MLA_ERR_INVALID_ARG;
    cudaError_t e = mla::launch_cache_write(latent, latent_stride, k_pe, k_pe_stride, slot_mapping, num_tokens, cache,
                                            num_slots, cache_kind, status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_gather_upconvert(const void* cache, int64_t num_slots, int page_size, const int32_t* block_table,
                         int64_t block_table_stride, const int32_t* cu_seq_lens, int B, int64_t num_rows, void* dst,
                         int64_t dst_stride, void* stream) {
    if (B < 0 || num_rows < 0 || page_size <= 0 || num_slots <= 0) return MLA_ERR_INVALID_ARG;
    if (B == 0 || num_rows == 0) return MLA_OK;
    if (!cache || !block_table || !cu_seq_lens || !dst) return MLA_ERR_INVALID_ARG;
    if (!aligned16(cache) || !aligned16(dst)) return MLA_ERR_INVALID_ARG;
    if (block_table_stride < 1 || dst_stride < mla::kW || dst_stride % 8) return MLA_ERR_INVALID_ARG;
    if (num_rows > (static_cast<int64_t>(UINT32_MAX) / 4) * 32) return MLA_ERR_UNSUPPORTED;  // grid size
    cudaError_t e = mla::launch_gather_upconvert(cache, num_slots, page_size, block_table, block_table_stride,
                                                 cu_seq_lens, B, num_rows, dst, dst_stride,
                                                 static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

size_t mla_decode_workspace_bytes(int B, int q_len, int Hq, int num_ctas) {
    if (B <= 0 || q_len <= 0 || Hq <= 0 || num_ctas < 0) return 0;
    int sms = 0;
    if (num_ctas == 0) {
        sms = mla_num_sms();
        if (sms <= 0) return 0;
    }
    return decode_ws_bytes(B, Hq * q_len, ws_ctas(num_ctas, sms));
}

}  // extern "C"

namespace {

// mla_decode and mla_decode_varlen: q_len is the (largest) verify length,
// cu_q null or the device prefix sums of per-request lengths, total_q the
// query tokens in q_lat / out (B * q_len for the uniform call).
int decode_impl(const void* q_lat, const void* q_pe, int64_t total_q, const void* cache, int cache_kind,
                int64_t num_slots, int page_size, const int32_t* block_table, int64_t block_table_stride,
                const int32_t* seq_lens, const int32_t* cu_q, int B, int q_len, int Hq, float scale, void* out,
                int out_dtype, float* lse, void* workspace, size_t workspace_bytes, int num_ctas, void* stream,
                int D = 512) {
    if (B <= 0 || q_len <= 0 || Hq <= 0 || page_size <= 0 || num_slots <= 0 || num_ctas < 0 || total_q <= 0)
        return MLA_ERR_INVALID_ARG;
    if (num_slots > 0x7fffffffLL) return MLA_ERR_UNSUPPORTED;  // TMA row coordinates are 32-bit
    if (cache_kind != MLA_CACHE_BF16_576 && cache_kind != MLA_CACHE_FP8_DS_MLA_656) return MLA_ERR_INVALID_ARG;
    if (out_dtype != MLA_OUT_BF16 && out_dtype != MLA_OUT_F32) return MLA_ERR_INVALID_ARG;
    if (!q_lat || !q_pe || !cache || !block_table || !seq_lens || !out || !lse || !workspace)
        return MLA_ERR_INVALID_ARG;
    if (!aligned16(q_lat) || !aligned16(q_pe) || !aligned16(cache) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return MLA_ERR_INVALID_ARG;
    if (block_table_stride < 1) return MLA_ERR_INVALID_ARG;
    const int64_t HQ64 = static_cast<int64_t>(Hq) * q_len;
    if (HQ64 > (1 << 20)) return MLA_ERR_UNSUPPORTED;
    const int HQ = static_cast<int>(HQ64);

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
    const DevInfo di = dev_info(dev);
    if (di.sms <= 0) return MLA_ERR_CUDA;
    if (di.major != 10) return MLA_ERR_UNSUPPORTED;
    const int GY = (HQ + 63) / 64;
    if (GY > 65535) return MLA_ERR_UNSUPPORTED;
    // TMA row coordinates of the queries are 32-bit
    if (total_q * Hq + 64 > INT32_MAX) return MLA_ERR_UNSUPPORTED;
    const int NP = rows_padded(HQ < 64 ? HQ : 64);
    // pages whose rows cannot be fetched as 8-row TMA boxes go through the
    // load/convert warps
    const bool lsu = (page_size % 8) != 0;
    // bf16 pools, and fp8 pools up to 64 query rows: folded 64-token tiles,
    // one CTA per worker (or a CTA pair, see decode_fold_ctas); fp8 pools
    // above 64 rows and odd page sizes: 128-token tiles split over clusters
    // of two CTAs
    const bool fold = !lsu && (cache_kind == MLA_CACHE_BF16_576 || mla::fold_supported(NP, D, cache_kind, GY));
    // other latent widths: bf16 rows of D + 64 values, folded tiles only
    if (D != 512 && (!fold || !mla::fold_supported(NP, D, cache_kind, GY))) return MLA_ERR_UNSUPPORTED;
    const int nctas = ws_ctas(num_ctas, di.sms);  // what the workspace holds records and slots for
    int W = fold ? mla::decode_fold_ctas(NP, D, cache_kind, GY, num_ctas)
                 : mla::decode_clusters(NP, lsu, cache_kind, num_ctas);
    if (W <= 0) return MLA_ERR_CUDA;
    W = std::min(W, (fold && !mla::fold_is_pair(D)) ? nctas : nctas / 2);
    const int tile = fold ? 64 : 128;
    const WsLayout wl = decode_ws_layout(B, HQ, nctas, D);
    if (workspace_bytes < wl.total) return MLA_ERR_WORKSPACE;

    // Two TMA descriptors over the pool [num_slots, 576] bf16: 64-dim latent
    // chunks (128-byte swizzle) and 32-dim rope halves (64-byte swizzle), both
    // gcd(page_size, tile) rows high so a box never crosses a page.
    mla::DecodeMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    CUtensorMap& tmap_lat = maps.lat;
    CUtensorMap& tmap_rope = maps.rope;
    auto enc = encode_fn();
    if (!enc) return MLA_ERR_CUDA;
    {
        // queries: q_lat [total_q * Hq, 512] and q_pe [total_q * Hq, 64] bf16, NP-row boxes
        const cuuint64_t rows = static_cast<cuuint64_t>(total_q) * Hq;
        cuuint64_t gq[2] = {static_cast<cuuint64_t>(D), rows};
        cuuint64_t sq[1] = {static_cast<cuuint64_t>(D) * 2};
        cuuint64_t gp[2] = {64u, rows};
        cuuint64_t sp[1] = {128u};
        cuuint32_t estride[2] = {1u, 1u};
        cuuint32_t bq[2] = {64u, static_cast<cuuint32_t>(NP)};
        cuuint32_t bp[2] = {32u, static_cast<cuuint32_t>(NP)};
        CUresult r = enc(&maps.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q_lat), gq, sq, bq, estride,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return MLA_ERR_CUDA;
        r = enc(&maps.qpe, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q_pe), gp, sp, bp, estride,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return MLA_ERR_CUDA;
    }
    if (!lsu) {
        // pool rows as 2-D tensors, gcd(page_size, tile) rows per box so a box
        // never crosses a page
        const int br = gcd_int(page_size, tile);
        const bool fp8 = cache_kind == MLA_CACHE_FP8_DS_MLA_656;
        const cuuint64_t row_bytes = fp8 ? mla::kRowFp8 : static_cast<cuuint64_t>(D + mla::kP) * 2;
        cuuint32_t estride[2] = {1u, 1u};
        CUresult r;
        if (!fp8) {
            cuuint64_t gdim[2] = {static_cast<cuuint64_t>(D + mla::kP), static_cast<cuuint64_t>(num_slots)};
            cuuint64_t gstride[1] = {row_bytes};
            cuuint32_t box_lat[2] = {64u, static_cast<cuuint32_t>(br)};
            r = enc(&tmap_lat, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(cache), gdim, gstride, box_lat,
                    estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) return MLA_ERR_CUDA;
        } else {
            // bytes of the 656-byte row: codes [0, 512), scales [512, 528)
            cuuint64_t gdim[2] = {row_bytes, static_cast<cuuint64_t>(num_slots)};
            cuuint64_t gstride[1] = {row_bytes};
            // folded tiles take 64 code bytes of a row per box (one K-block's
            // half), the cluster kernel 256 (a CTA's half of the row)
            cuuint32_t box_codes[2] = {fold ? 64u : 256u, static_cast<cuuint32_t>(br)};
            cuuint32_t box_scales[2] = {16u, static_cast<cuuint32_t>(br)};
            r = enc(&tmap_lat, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(cache), gdim, gstride, box_codes,
                    estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) return MLA_ERR_CUDA;
            r = enc(&maps.aux, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(cache), gdim, gstride, box_scales,
                    estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) return MLA_ERR_CUDA;
        }
        // rope: the row as bf16 elements; the rope halves at element 512 (bf16)
        // or 264 (fp8: byte 528), 32 values each
        cuuint64_t gdim[2] = {row_bytes / 2, static_cast<cuuint64_t>(num_slots)};
        cuuint64_t gstride[1] = {row_bytes};
        cuuint32_t box_rope[2] = {32u, static_cast<cuuint32_t>(br)};
        r = enc(&tmap_rope, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(cache), gdim, gstride, box_rope,
                estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return MLA_ERR_CUDA;
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* ws = static_cast<uint8_t*>(workspace);

    mla::DecodeParams p;
    p.q_lat = static_cast<const __nv_bfloat16*>(q_lat);
    p.q_pe = static_cast<const __nv_bfloat16*>(q_pe);
    p.cache = static_cast<const uint8_t*>(cache);
    p.num_slots = num_slots;
    p.block_table = block_table;
    p.bt_stride = block_table_stride;
    p.seq_lens = seq_lens;
    p.out = out;
    p.lse = lse;
    p.status = reinterpret_cast<int*>(ws);
    p.rec = reinterpret_cast<int*>(ws + wl.rec_off);
    p.part_lse = reinterpret_cast<float*>(ws + wl.lse_off);
    p.part_o = reinterpret_cast<float*>(ws + wl.o_off);
    p.scale_log2 = scale * 1.4426950408889634f;
    p.page_size = page_size;
    p.run_rows = gcd_int(page_size, tile);
    p.tile_shift = fold ? 6 : 7;
    p.B = B;
    p.Qt = q_len;
    p.Hq = Hq;
    p.HQ = HQ;
    p.out_f32 = out_dtype == MLA_OUT_F32;
    p.SPG = W + B;
    // what a request boundary costs a worker, in tiles (measured on the
    // cluster kernel: about one and a half 128-token tiles at 16 query rows;
    // the 64-row drain is four times larger; folded tiles are half as long;
    // at 64 rows the folded kernel drains a finished segment before the next
    // one's first value product, about two tiles' time)
    p.wseg = fold ? (NP == 16 ? 4 : NP == 32 ? 8 : 4) : (NP == 16 ? 2 : NP == 32 ? 4 : 8);
    p.test_hold = g_test_hold.exchange(0);
    p.cu_q = cu_q;
    p.total_q = static_cast<int>(total_q);  // total_q * Hq < 2^31 (checked above)
    p.lat_dim = D;
    p.rope_dim = mla::kP;
    cudaError_t e = fold ? mla::launch_decode_fold(maps, p, NP, cache_kind, W, GY, s)
                         : mla::launch_decode(maps, p, NP, lsu, cache_kind, W, GY, s);
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace

extern "C" {

int mla_decode(const void* q_lat, const void* q_pe, const void* cache, int cache_kind, int64_t num_slots,
               int page_size, const int32_t* block_table, int64_t block_table_stride, const int32_t* seq_lens, int B,
               int q_len, int Hq, float scale, void* out, int out_dtype, float* lse, void* workspace,
               size_t workspace_bytes, int num_ctas, void* stream) {
    if (B <= 0 || q_len <= 0) return MLA_ERR_INVALID_ARG;
    return decode_impl(q_lat, q_pe, static_cast<int64_t>(B) * q_len, cache, cache_kind, num_slots, page_size,
                       block_table, block_table_stride, seq_lens, nullptr, B, q_len, Hq, scale, out, out_dtype, lse,
                       workspace, workspace_bytes, num_ctas, stream);
}

size_t mla_decode_latent_workspace_bytes(int B, int q_len, int Hq, int lat_dim, int num_ctas) {
    if (B <= 0 || q_len <= 0 || Hq <= 0 || num_ctas < 0 || lat_dim <= 0 || lat_dim % 128) return 0;
    int sms = 0;
    if (num_ctas == 0) {
        sms = mla_num_sms();
        if (sms <= 0) return 0;
    }
    return decode_ws_bytes(B, Hq * q_len, ws_ctas(num_ctas, sms), lat_dim);
}

int mla_cache_write_latent(const void* latent, int64_t latent_stride, const void* k_pe, int64_t k_pe_stride,
                           const int64_t* slot_mapping, int64_t num_tokens, void* cache, int64_t num_slots,
                           int lat_dim, int32_t* status, void* stream) {
    if (num_tokens < 0 || num_slots < 0) return MLA_ERR_INVALID_ARG;
    if (lat_dim != 256 && lat_dim != 512 && lat_dim != 768 && lat_dim != 1792) return MLA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return MLA_OK;
    if (!latent || !k_pe || !slot_mapping || !cache) return MLA_ERR_INVALID_ARG;
    if (!aligned16(latent) || !aligned16(k_pe) || !aligned16(cache)) return MLA_ERR_INVALID_ARG;
    if (latent_stride < lat_dim || latent_stride % 8 || k_pe_stride < mla::kP || k_pe_stride % 8)
        return MLA_ERR_INVALID_ARG;
    if (status && (reinterpret_cast<uintptr_t>(status) & 3u)) return MLA_ERR_INVALID_ARG;
    cudaError_t e = mla::launch_cache_write_latent(latent, latent_stride, k_pe, k_pe_stride, slot_mapping, num_tokens,
                                                   cache, num_slots, lat_dim, status,
                                                   static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_decode_latent(const void* q_lat, const void* q_pe, const void* cache, int lat_dim, int64_t num_slots,
                      int page_size, const int32_t* block_table, int64_t block_table_stride, const int32_t* seq_lens,
                      int B, int q_len, int Hq, float scale, void* out, int out_dtype, float* lse, void* workspace,
                      size_t workspace_bytes, int num_ctas, void* stream) {
    if (B <= 0 || q_len <= 0) return MLA_ERR_INVALID_ARG;
    if (lat_dim != 256 && lat_dim != 512 && lat_dim != 768 && lat_dim != 1792) return MLA_ERR_UNSUPPORTED;
    return decode_impl(q_lat, q_pe, static_cast<int64_t>(B) * q_len, cache, MLA_CACHE_BF16_576, num_slots, page_size,
                       block_table, block_table_stride, seq_lens, nullptr, B, q_len, Hq, scale, out, out_dtype, lse,
                       workspace, workspace_bytes, num_ctas, stream, lat_dim);
}

int mla_decode_varlen(const void* q_lat, const void* q_pe, int64_t total_q_tokens, const void* cache,
                      int cache_kind, int64_t num_slots, int page_size, const int32_t* block_table,
                      int64_t block_table_stride, const int32_t* seq_lens, const int32_t* cu_q_lens, int B,
                      int max_q_len, int Hq, float scale, void* out, int out_dtype, float* lse, void* workspace,
                      size_t workspace_bytes, int num_ctas, void* stream) {
    if (!cu_q_lens) return MLA_ERR_INVALID_ARG;
    return decode_impl(q_lat, q_pe, total_q_tokens, cache, cache_kind, num_slots, page_size, block_table,
                       block_table_stride, seq_lens, cu_q_lens, B, max_q_len, Hq, scale, out, out_dtype, lse,
                       workspace, workspace_bytes, num_ctas, stream);
}

int mla_decode_static_scratch(const void* q_lat, const void* q_pe, const void* cache, int cache_kind,
                              int64_t num_slots, int page_size, const int32_t* block_table,
                              int64_t block_table_stride, const int32_t* seq_lens, int B, int q_len, int Hq,
                              float scale, void* out, int out_dtype, float* lse, int num_ctas, void* stream) {
    const size_t need = mla_decode_workspace_bytes(B, q_len, Hq, num_ctas);
    if (need == 0) return MLA_ERR_INVALID_ARG;
    if (need > MLA_STATIC_SCRATCH_BYTES) return MLA_ERR_SCRATCH_LIMIT;
    void* scratch = decode_scratch_ptr();
    if (!scratch) return MLA_ERR_CUDA;
    return mla_decode(q_lat, q_pe, cache, cache_kind, num_slots, page_size, block_table, block_table_stride,
                      seq_lens, B, q_len, Hq, scale, out, out_dtype, lse, scratch, MLA_STATIC_SCRATCH_BYTES,
                      num_ctas, stream);
}

int mla_static_scratch_status(int32_t* dst, int n, void* stream) {
    if (!dst || n < 1 || n > 12) return MLA_ERR_INVALID_ARG;
    void* scratch = decode_scratch_ptr();
    if (!scratch) return MLA_ERR_CUDA;
    cudaError_t e = cudaMemcpyAsync(dst, scratch, static_cast<size_t>(n) * sizeof(int32_t), cudaMemcpyDefault,
                                    static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

void mla_test_hold_next_decode(void) { g_test_hold.store(1); }

void mla_test_slow_pv_next_decode(void) { g_test_hold.store(2); }

int mla_merge_lse(const float* part_out, const float* part_lse, int S, int64_t N, void* out, int out_dtype,
                  float* lse, void* stream) {
    if (S < 0 || N < 0) return MLA_ERR_INVALID_ARG;
    if (out_dtype != MLA_OUT_BF16 && out_dtype != MLA_OUT_F32) return MLA_ERR_INVALID_ARG;
    if (N == 0) return MLA_OK;
    if ((S > 0 && (!part_out || !part_lse)) || !out) return MLA_ERR_INVALID_ARG;
    if ((S > 0 && !aligned16(part_out)) || !aligned16(out)) return MLA_ERR_INVALID_ARG;
    cudaError_t e = mla::launch_merge_lse(part_out, part_lse, S, N, out, out_dtype == MLA_OUT_F32, lse,
                                          static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // extern "C"
