// C ABI of the library: argument validation, the shape planner, tensor-map
// encoding, the nvfp4_gemm scale workspace, the device status word.
// Declarations and their contracts are in include/bsgemm.h.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>
#include <string>

#include "bsg_internal.h"
#include "bsgemm.h"
#include "group.cuh"

// Device status word written by bounded waits that run out (one per device).
__device__ unsigned int g_bsg_status_word;

namespace {

using bsg::GemmArgs;
using bsg::GemmMaps;
using bsg::Kind;
using bsg::PlanInfo;

constexpr unsigned long long kDefaultWatchdogNs = 1000000000ull;
constexpr int kMaxDevices = 64;

std::atomic<unsigned long long> g_watchdog_ns{kDefaultWatchdogNs};
// M tiles per rasterisation group (L2 reuse of B). Swept on GB300 over 1..32:
// 16 beat 8 on every alternating repeat (FP8 8192^3 +2.1 %, NVFP4 16384^3
// +0.9 %); L2-resident shapes do not depend on it.
constexpr int kDefaultRasterGroup = 16;
std::atomic<int> g_raster_group{kDefaultRasterGroup};
std::atomic<int> g_pdl{0};              // programmatic dependent launch (off by default)
std::mutex g_mu;
int g_forced_plan = -1;                 // guarded by g_mu
thread_local uint32_t t_last_status_word = 0;
thread_local int t_last_launches = 0;
thread_local const char *t_last_plan = "";      // plan of the last GEMM launch on this thread

struct DeviceState {
    bool init = false;
    int rc = BSG_OK;
    int sms = 0;
    unsigned int *status = nullptr;     // device address of g_bsg_status_word
    uint8_t *ws = nullptr;              // nvfp4_gemm scale workspace
    size_t ws_bytes = 0;
};
DeviceState g_dev[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// State of the current device, initialised once: compute capability check,
// SM count, status-word address.
int current_device(DeviceState **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return BSG_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &d = g_dev[dev];
    if (!d.init) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            d.rc = BSG_ERR_CUDA;
        } else if (major != 10 || minor != 3) {
            d.rc = BSG_ERR_UNSUPPORTED_DEVICE;
        } else if (cudaGetSymbolAddress(reinterpret_cast<void **>(&d.status), g_bsg_status_word) !=
                   cudaSuccess) {
            d.rc = BSG_ERR_CUDA;
        } else {
            d.rc = BSG_OK;
        }
        d.init = true;
    }
    *out = &d;
    return d.rc;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t swizzled_bytes(int rows, int K)
{
    if (rows < 1 || K < 16 || (K % 16) != 0)
        return 0;
    const size_t pr = ((size_t)rows + 127u) / 128u * 128u;
    const size_t pc = ((size_t)(K / 16) + 3u) / 4u * 4u;
    return pr * pc;
}

// Planner: the default plan for a shape; -1 if none fits. The rules follow
// CUDA-graph timings of every plan and split on the skinny cells (M 64..512
// x N 3072 / 12288 x K 3072 / 12288, cold L2) and the square sizes:
//   * NVFP4, the swap-AB split-K kernel when the weight tiles leave room to
//     split K at least in two with the whole grid resident (N/128 tiles x 2
//     <= SMs): for M <= 64 (the 3-stage ring up to K = 4096, where a CTA
//     streams a few k-blocks, else the 6-stage one), and up to 256
//     activation rows for long K (>= 8192), where streaming the weights
//     dominates its fixed costs;
//   * 129..512 activation rows with 256 x 256 pair tiles enough to give
//     every SM a quarter of one (M/256 x N/256 x 4 >= SMs): the CTA pair,
//     whose tile moves half the bytes per FLOP of a 1-SM 128 x 128 tile;
//   * otherwise, while 128 x 128 output tiles number at most 4 per SM, the
//     1-SM 128 x 128 kernel (more CTAs in flight than 256-wide tiles);
//   * M <= 128 beyond that: the 1-SM 128 x 256 kernel; larger M: the CTA
//     pair (256 x 128 for N <= 128, else 256 x 256; FP8 256 x 512 where N
//     is a multiple of 512).
int default_plan(Kind kind, int M, int N, int K, int num_sms)
{
    const char *name = nullptr;
    const long long tiles128 = (long long)((M + 127) / 128) * (long long)((N + 127) / 128);
    const bool few_tiles = tiles128 <= 4LL * num_sms;
    if (kind == Kind::NVFP4) {
        const int weight_tiles = (N + 127) / 128;
        const bool can_split = 2 * weight_tiles <= num_sms && K >= 512;
        const long long pair_tiles = (long long)((M + 255) / 256) * (long long)((N + 255) / 256);
        if (can_split && (M <= 64 || (M <= 256 && K >= 8192)))
            name = M <= 64 ? (K <= 4096 ? "nvfp4_skinny_m64_s3" : "nvfp4_skinny_m64_s6")
                           : M <= 128 ? "nvfp4_skinny_m128_s3" : "nvfp4_skinny_m256_s4";
        else if (M > 128 && M <= 512 && N > 128 && 4 * pair_tiles >= num_sms)
            name = "nvfp4_tc2_256x256_s5_acc1";
        else if (few_tiles || N <= 128)
            name = M <= 128 || few_tiles ? "nvfp4_tc1_128x128_s5_acc2" : "nvfp4_tc2_256x128_s6_acc2";
        else
            name = M <= 128 ? "nvfp4_tc1_128x256_s3_acc1" : "nvfp4_tc2_256x256_s5_acc1";
    } else if (kind == Kind::NVFP4_BF16) {
        // expanded A staged in TMEM (5 or 8 stages) measured 1.2x the
        // shared-memory expansion (3 or 5 stages), and the 1-SM 128 x 256
        // tile 1.1x the CTA-pair 256 x 256 one (8 stages); 128 x 128 tiles
        // only where N leaves no 256-wide tile
        name = N <= 128 ? "nvfp4bf16_tc1_128x128_s8_acc2_tmema" : "nvfp4bf16_tc1_128x256_s5_acc1_tmema";
    } else {
        // FP8 pair tiles 512 wide where N is whole 512-column tiles: each
        // SM's 128 rows of B in one copy of two 128-row halves, one
        // accumulator filling TMEM; 2.4-6.4 % faster than 256-wide tiles
        // from 2048 x 4096 x 8192 to 16384^3, bit-identical
        const bool small_m = M <= 128;   // a 256-row pair tile would idle half its SMs
        if (small_m)
            name = N <= 128 ? "fp8_tc1_128x128_s6_acc2" : "fp8_tc1_128x256_s4_acc2";
        else if (N % 512 == 0)
            name = "fp8_tc2_256x512_s4_acc1";
        else
            name = N <= 128 ? "fp8_tc1_128x128_s6_acc2" : "fp8_tc2_256x256_s6_acc2";
    }
    return bsg::find_plan(name);
}

// Activation rows a skinny plan serves: one block of tile_m rows, or two
// where a block is whole 128-row scale blocks.
int skinny_max_rows(const PlanInfo &pi) { return pi.tile_m >= 128 ? 2 * pi.tile_m : pi.tile_m; }

int choose_plan(Kind kind, int M, int N, int K, int num_sms, int *plan)
{
    int forced;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        forced = g_forced_plan;
    }
    if (forced >= 0) {
        const PlanInfo &fp = bsg::plan_info(forced);
        // a tile-packed plan reads operands only nvfp4_gemm_packed supplies
        if (fp.kind != kind || fp.packed || (fp.family == bsg::Family::SKINNY && M > skinny_max_rows(fp)) ||
            (fp.bn == 512 && (N % 256) != 0))
            return BSG_ERR_NO_PLAN;
        *plan = forced;
        return BSG_OK;
    }
    *plan = default_plan(kind, M, N, K, num_sms);
    return *plan >= 0 ? BSG_OK : BSG_ERR_NO_PLAN;
}

// Everything a tiled tensor map is encoded from (the other encode
// arguments are fixed: unit element strides, no interleave, 256-byte L2
// promotion, zero fill). Unused dimensions are zero; the struct is cleared
// byte by byte before it is filled, so keys compare with memcmp.
struct MapKey {
    const void *ptr;
    uint64_t dims[3];
    uint64_t strides[2];
    uint32_t box[3];
    int32_t dtype, rank, swizzle, zero;
};

// The last kMapCacheSize maps this thread encoded: a map is a pure function
// of its key, so a repeated call (the same buffers and shape, the usual case
// for a layer run again) copies the 128 bytes instead of encoding them.
constexpr int kMapCacheSize = 32;
struct MapCacheEntry {
    MapKey key;
    CUtensorMap map;
};
thread_local MapCacheEntry t_maps[kMapCacheSize];
thread_local int t_maps_used = 0;
thread_local int t_maps_next = 0;

int encode_tiled(CUtensorMap *map, CUtensorMapDataType dtype, int rank, const void *ptr, const uint64_t *dims,
                 const uint64_t *strides, const uint32_t *box, CUtensorMapSwizzle swizzle)
{
    MapKey key;
    std::memset(&key, 0, sizeof key);
    key.ptr = ptr;
    for (int i = 0; i < rank; ++i) {
        key.dims[i] = dims[i];
        key.box[i] = box[i];
    }
    for (int i = 0; i + 1 < rank; ++i)
        key.strides[i] = strides[i];
    key.dtype = (int32_t)dtype;
    key.rank = rank;
    key.swizzle = (int32_t)swizzle;
    for (int i = 0; i < t_maps_used; ++i)
        if (std::memcmp(&t_maps[i].key, &key, sizeof key) == 0) {
            *map = t_maps[i].map;
            return BSG_OK;
        }
    auto fn = encode_fn();
    if (!fn)
        return BSG_ERR_CUDA;
    cuuint64_t d[3], st[2];
    cuuint32_t b[3], es[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
    }
    for (int i = 0; i + 1 < rank; ++i)
        st[i] = strides[i];
    CUresult r = fn(map, dtype, (cuuint32_t)rank, const_cast<void *>(ptr), d, st, b, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return BSG_ERR_CUDA;
    MapCacheEntry &e = t_maps[t_maps_next];
    e.key = key;
    e.map = *map;
    t_maps_next = (t_maps_next + 1) % kMapCacheSize;
    if (t_maps_used < kMapCacheSize)
        ++t_maps_used;
    return BSG_OK;
}

int encode_2d(CUtensorMap *map, CUtensorMapDataType dtype, const void *ptr, uint64_t inner,
              uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B)
{
    const uint64_t dims[2] = {inner, outer};
    const uint64_t strides[1] = {row_bytes};
    const uint32_t box[2] = {box_inner, box_outer};
    return encode_tiled(map, dtype, 2, ptr, dims, strides, box, swizzle);
}

// A 3-D view: inner x mid x outer elements, byte strides of mid and outer.
int encode_3d(CUtensorMap *map, const void *ptr, uint64_t inner, uint64_t mid, uint64_t outer, uint64_t mid_stride,
              uint64_t outer_stride, uint32_t box_inner, uint32_t box_mid, uint32_t box_outer,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE)
{
    const uint64_t dims[3] = {inner, mid, outer};
    const uint64_t strides[2] = {mid_stride, outer_stride};
    const uint32_t box[3] = {box_inner, box_mid, box_outer};
    return encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, ptr, dims, strides, box, swizzle);
}

// Resident clusters of `splits` CTAs (1..8) for skinny plan id on the
// current device (cached).
int skinny_cluster_capacity(int id, int splits)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices || id < 0 || id >= 8 || splits < 1 ||
        splits > 8)
        return 0;
    static int cache[kMaxDevices][8][9] = {};
    std::lock_guard<std::mutex> lk(g_mu);
    if (cache[dev][id][splits] == 0)
        cache[dev][id][splits] = bsg::skinny_max_clusters(id, splits);
    return cache[dev][id][splits];
}

// K splits of the skinny kernel (a cluster of that many CTAs per weight tile
// and activation block); 0 = chosen per call.
std::atomic<int> g_skinny_splits{0};

// The split count of a skinny launch: among the splits S the plan takes, S
// <= k-blocks whose clusters all fit on the device at once, the one whose
// busiest SM streams the fewest k-blocks (CTAs per SM x k-blocks per CTA),
// ties going to the smaller S (less to exchange).
int skinny_splits(int id, int mask, int units, int num_k_blocks, int num_sms)
{
    int best = 1;
    long long best_cost = -1;
    for (int s = 1; s <= 8; ++s) {
        if (!(mask & (1 << s)) || s > num_k_blocks || units > skinny_cluster_capacity(id, s))
            continue;
        const long long ctas = (long long)units * s;
        const long long cost = (ctas + num_sms - 1) / num_sms * ((num_k_blocks + s - 1) / s);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = s;
        }
    }
    return best;
}

// Epilogue operands of one call (all null: the plain GEMM).
struct Epilogue {
    const float *bias = nullptr;
    const float *gamma = nullptr;
    const int32_t *scatter = nullptr;
    int m_out = 0;
};

void set_epilogue(GemmArgs &a, const Epilogue &e, void *D)
{
    a.bias = e.bias;
    a.gamma = e.gamma;
    a.scatter = e.scatter;
    a.d = static_cast<uint16_t *>(D);
    a.m_out = e.m_out;
}

int run_skinny(int plan, const PlanInfo &pi, int M, int N, int K, const void *A, const void *B,
               const uint8_t *sfa, const uint8_t *sfb, float alpha, void *D, const Epilogue &epi,
               cudaStream_t stream, DeviceState *ds);

// Rows of D: M, or m_out when rows are scattered (the tensor map of D then
// only describes the buffer; the scattered rows are stored without it).
uint64_t d_rows(int M, const Epilogue &e) { return (uint64_t)(e.scatter ? e.m_out : M); }

// Swap-AB split-K launch for skinny M: weight tiles of 128 rows on grid x,
// the K split on grid y (one thread-block cluster per weight tile).
int run_skinny(int plan, const PlanInfo &pi, int M, int N, int K, const void *A, const void *B,
               const uint8_t *sfa, const uint8_t *sfb, float alpha, void *D, const Epilogue &epi,
               cudaStream_t stream, DeviceState *ds)
{
    const int id = plan - bsg::tc1_num_plans() - bsg::pair_num_plans();
    const int num_n_tiles = (N + pi.bn - 1) / pi.bn;
    const int num_k_blocks = K / pi.k_block;
    const int halves = (M + pi.tile_m - 1) / pi.tile_m;      // activation blocks (1, or 2 for tile_m >= 128)
    const int forced = g_skinny_splits.load();
    const int splits = forced > 0 ? forced
                                  : skinny_splits(id, pi.splits_mask, num_n_tiles * halves, num_k_blocks, ds->sms);
    if (!(pi.splits_mask & (1 << splits)) || splits > num_k_blocks ||
        num_n_tiles * halves > skinny_cluster_capacity(id, splits))
        return BSG_ERR_NO_PLAN;
    const uint64_t row_bytes = (uint64_t)K / 2u;
    GemmMaps maps;
    std::memset(&maps, 0, sizeof maps);
    int rc;
    if ((rc = encode_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, row_bytes, (uint64_t)M, row_bytes,
                        128, (uint32_t)pi.tile_m)) != BSG_OK ||
        (rc = encode_2d(&maps.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, row_bytes, (uint64_t)N, row_bytes,
                        128, (uint32_t)pi.bn)) != BSG_OK)
        return rc;
    GemmArgs a;
    std::memset(&a, 0, sizeof a);
    a.M = M;
    a.N = N;
    a.K = K;
    a.num_m_tiles = 1;
    a.num_n_tiles = num_n_tiles;
    a.num_k_blocks = num_k_blocks;
    a.raster_group = 1;
    a.sf_col_blocks = (K / 16 + 3) / 4;
    a.sfb_row_blocks = (N + 127) / 128;
    a.sfx_row_blocks = (M + 127) / 128;
    a.sfa = sfa;
    a.sfb = sfb;
    a.alpha = alpha;
    a.status = ds->status;
    a.timeout_ns = g_watchdog_ns.load();
    set_epilogue(a, epi, D);
    a.pdl = g_pdl.load();
    if (bsg::skinny_launch(id, maps, a, splits, halves, stream) != cudaSuccess)
        return BSG_ERR_CUDA;
    ++t_last_launches;
    t_last_plan = pi.name;
    return BSG_OK;
}

// Encode the maps and launch one persistent GEMM.
int run_gemm(Kind kind, int M, int N, int K, const void *A, const void *B, const uint8_t *sfa,
             const uint8_t *sfb, const float *sA, const float *sB, float alpha, void *D,
             cudaStream_t stream, DeviceState *ds, const Epilogue &epi = Epilogue(), bool b_f16 = false,
             const uint8_t *a_packed = nullptr, const uint8_t *b_packed = nullptr)
{
    int plan = -1;
    int rc = BSG_OK;
    const bool packed = a_packed != nullptr;
    if (packed)
        plan = bsg::find_plan("nvfp4_tc2_256x256_s5_acc1_packed");   // the one tile-packed plan
    else if ((rc = choose_plan(kind, M, N, K, ds->sms, &plan)) != BSG_OK)
        return rc;
    if (plan < 0)
        return BSG_ERR_NO_PLAN;
    const PlanInfo &pi = bsg::plan_info(plan);
    const bool dense = kind == Kind::NVFP4_BF16;
    // bytes per row: packed E2M1 (K/2), E4M3 (K), or for the dense kind packed
    // A and BF16 B (2K)
    const uint64_t row_bytes = kind == Kind::FP8 ? (uint64_t)K : (uint64_t)K / 2u;
    const uint64_t b_row_bytes = dense ? 2u * (uint64_t)K : row_bytes;
    if (pi.family == bsg::Family::SKINNY)
        return run_skinny(plan, pi, M, N, K, A, B, sfa, sfb, alpha, D, epi, stream, ds);

    GemmMaps maps;
    std::memset(&maps, 0, sizeof maps);
    // A: 128 rows per CTA (dense: 32 bytes of codes per row and stage,
    // unswizzled, expanded in shared memory); B: the CTA's share of the
    // tile's N rows, 128 bytes per row and stage
    // (tile-packed plans load A and B by bulk copies and read neither map,
    // which then repeat D's)
    if (packed) {
        if ((rc = encode_2d(&maps.d, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, (uint64_t)N, d_rows(M, epi),
                            (uint64_t)N * 2u, 64, 32)) != BSG_OK)
            return rc;
        maps.a = maps.d;
        maps.b = maps.d;
    } else if ((rc = encode_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, row_bytes, (uint64_t)M, row_bytes,
                        dense ? 32 : 128, 128u,
                        dense ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B)) != BSG_OK ||
        (rc = encode_2d(&maps.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, b_row_bytes, (uint64_t)N, b_row_bytes,
                        128, (uint32_t)(pi.bn / pi.cta_group))) != BSG_OK ||
        (rc = encode_2d(&maps.d, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, (uint64_t)N, d_rows(M, epi),
                        (uint64_t)N * 2u, 64, 32)) != BSG_OK)
        return rc;
    if (pi.bn == 512) {
        // FP8 tiles 512 wide: each CTA's 128 rows of both 256-row halves of
        // the tile in one copy -- a 3-D view (K bytes, rows of a half,
        // halves; N a multiple of 256 so the halves tile B exactly)
        if ((rc = encode_3d(&maps.b, B, b_row_bytes, 256, (uint64_t)N / 256u, b_row_bytes, 256u * b_row_bytes, 128,
                            128, 2, CU_TENSOR_MAP_SWIZZLE_128B)) != BSG_OK)
            return rc;
    }
    if (pi.cta_group == 2 && kind == Kind::NVFP4) {
        // swizzled scales viewed as rows of 256 bytes; one stage = 8 rows
        if ((rc = encode_2d(&maps.sfa, CU_TENSOR_MAP_DATA_TYPE_UINT8, sfa, 256,
                            swizzled_bytes(M, K) / 256u, 256, 256, 8, CU_TENSOR_MAP_SWIZZLE_NONE)) !=
                BSG_OK ||
            // B's: 256-byte rows x (rows of one 128-row block) x row blocks,
            // so that one copy takes a stage's blocks of all the tile's rows
            (rc = encode_3d(&maps.sfb, sfb, 256, (uint64_t)K / 32u, ((uint64_t)N + 127u) / 128u, 256,
                            (uint64_t)K / 32u * 256u, 256, 8, (uint32_t)(pi.bn / 256 > 0 ? 2 : 1))) !=
                BSG_OK)
            return rc;
    } else {
        maps.sfa = maps.a;
        maps.sfb = maps.a;
    }

    GemmArgs a;
    std::memset(&a, 0, sizeof a);
    a.M = M;
    a.N = N;
    a.K = K;
    a.num_m_tiles = (M + pi.tile_m - 1) / pi.tile_m;
    a.num_n_tiles = (N + pi.bn - 1) / pi.bn;
    a.num_k_blocks = K / pi.k_block;
    a.raster_group = g_raster_group.load();   // M tiles per rasterisation group (L2 reuse of B)
    a.b_f16 = b_f16 ? 1 : 0;
    a.sf_col_blocks = (K / 16 + 3) / 4;
    a.sfb_row_blocks = (N + 127) / 128;
    a.sfa = sfa;
    a.sfb = sfb;
    a.a_packed = a_packed;
    a.b_packed = b_packed;
    a.alpha = alpha;
    a.sA = sA;
    a.sB = sB;
    a.status = ds->status;
    a.timeout_ns = g_watchdog_ns.load();
    set_epilogue(a, epi, D);
    a.pdl = g_pdl.load();
    // scheduling units: a tile per CTA or pair; the grid is a whole number
    // of clusters
    const long long units = (long long)a.num_m_tiles * a.num_n_tiles;
    const long long ctas = units * pi.cta_group;
    const int resident = bsg::max_resident_ctas(plan, ds->sms);
    if (resident < pi.cta_group)
        return BSG_ERR_CUDA;
    const int grid = (int)(ctas < resident ? ctas : resident);
    cudaError_t e = bsg::launch_gemm(plan, maps, a, grid, stream);
    if (e != cudaSuccess)
        return BSG_ERR_CUDA;
    ++t_last_launches;
    t_last_plan = pi.name;
    return BSG_OK;
}

// Grouped (ragged) NVFP4 GEMM: the 1-SM kernel's grouped instantiation, one
// 128-row tile row per 128 rows of each slice, or the CTA pair's (above).
// The slice table is built on the device from offs, so the grid is sized
// for the bound on the tile rows, ceil(M/128) + E; CTAs past the actual
// tiles exit at once.
// True for the dense (NVFP4 x 16-bit) plans the grouped GEMM runs: A staged
// in TMEM, and room beside the ring for the slice table.
static bool grouped_dense_plan(const PlanInfo &pi)
{
    const size_t n = std::strlen(pi.name);
    return pi.kind == Kind::NVFP4_BF16 && pi.family == bsg::Family::TC1 && n > 6 &&
           std::strcmp(pi.name + n - 6, "_tmema") == 0 && pi.smem_bytes + bsg::kGroupTableBytes <= 232448;
}

// The grouped mode of the CTA pair (NVFP4, up to kPairMaxGroups slices):
// one 256-row pair tile row per 256 rows of each slice, so the ~128-row
// slices of a routed MoE layer stream each weight tile once, half into each
// SM of the pair. Grid: the bound ceil(M/256) + E on the tile rows.
bool grouped_pair_plan(const PlanInfo &pi, int E)
{
    return E <= bsg::kPairMaxGroups && std::strcmp(pi.name, "nvfp4_tc2_256x256_s5_acc1") == 0;
}

int run_grouped_pair(int plan, int E, int M, int N, int K, const void *A, const uint8_t *sfa, const void *B,
                     const uint8_t *sfb, const int32_t *offs, float alpha, const Epilogue &epi, void *D,
                     cudaStream_t stream, DeviceState *ds)
{
    const PlanInfo &pi = bsg::plan_info(plan);
    const long long pt_bound = (long long)(M + 255) / 256 + E;
    const uint64_t row_bytes = (uint64_t)K / 2u;
    const uint64_t nrb = ((uint64_t)N + 127u) / 128u;       // 128-row scale blocks of one slice's weights
    const size_t sfa_bytes = ((size_t)(M + 127) / 128u + (size_t)E) * 128u * ((size_t)(K / 16 + 3) / 4u * 4u);
    GemmMaps maps;
    std::memset(&maps, 0, sizeof maps);
    int rc;
    if ((rc = encode_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, row_bytes, (uint64_t)M, row_bytes, 128,
                        128u)) != BSG_OK ||
        (rc = encode_2d(&maps.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, row_bytes, (uint64_t)E * (uint64_t)N,
                        row_bytes, 128, (uint32_t)(pi.bn / 2))) != BSG_OK ||
        (rc = encode_2d(&maps.d, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, (uint64_t)N, d_rows(M, epi),
                        (uint64_t)N * 2u, 64, 32)) != BSG_OK ||
        // the per-slice swizzled A scales as 256-byte rows; the E slices'
        // swizzled weight scales as one 3-D view whose row blocks run
        // through all slices (slice e's first block is e * nrb)
        (rc = encode_2d(&maps.sfa, CU_TENSOR_MAP_DATA_TYPE_UINT8, sfa, 256, sfa_bytes / 256u, 256, 256, 8,
                        CU_TENSOR_MAP_SWIZZLE_NONE)) != BSG_OK ||
        (rc = encode_3d(&maps.sfb, sfb, 256, (uint64_t)K / 32u, (uint64_t)E * nrb, 256, (uint64_t)K / 32u * 256u,
                        256, 8, 2)) != BSG_OK)
        return rc;
    GemmArgs a;
    std::memset(&a, 0, sizeof a);
    a.M = M;
    a.N = N;
    a.K = K;
    a.num_m_tiles = (int)pt_bound;      // bound only: the kernel counts the slices' tile rows
    a.num_n_tiles = (N + pi.bn - 1) / pi.bn;
    a.num_k_blocks = K / pi.k_block;
    a.raster_group = g_raster_group.load();
    a.sf_col_blocks = (K / 16 + 3) / 4;
    a.sfb_row_blocks = (int)nrb;
    a.sfa = sfa;
    a.sfb = sfb;
    a.alpha = alpha;
    a.status = ds->status;
    a.timeout_ns = g_watchdog_ns.load();
    set_epilogue(a, epi, D);
    a.num_groups = E;
    a.group_offs = offs;
    a.sfb_group_bytes = swizzled_bytes(N, K);
    a.pdl = g_pdl.load();
    const long long ctas = pt_bound * a.num_n_tiles * 2;
    const int resident = bsg::max_resident_ctas(plan, ds->sms);
    if (resident < 2)
        return BSG_ERR_CUDA;
    const int grid = (int)(ctas < resident ? ctas : resident);
    if (bsg::launch_gemm(plan, maps, a, grid, stream) != cudaSuccess)
        return BSG_ERR_CUDA;
    ++t_last_launches;
    t_last_plan = pi.name;
    return BSG_OK;
}

// dense: the right-hand sides are 16-bit (BF16, or FP16 with b_f16) [E][N][K]
int run_grouped(int E, int M, int N, int K, const void *A, const uint8_t *sfa, const void *B,
                const uint8_t *sfb, const int32_t *offs, float alpha, const Epilogue &epi, void *D,
                cudaStream_t stream, DeviceState *ds, bool dense = false, bool b_f16 = false)
{
    const long long mt_bound = (long long)(M + 127) / 128 + E;
    int plan;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        plan = g_forced_plan;
    }
    if (plan >= 0) {
        const PlanInfo &fp = bsg::plan_info(plan);
        if (!dense && grouped_pair_plan(fp, E))
            return run_grouped_pair(plan, E, M, N, K, A, sfa, B, sfb, offs, alpha, epi, D, stream, ds);
        if (dense ? !grouped_dense_plan(fp) : (fp.kind != Kind::NVFP4 || fp.family != bsg::Family::TC1))
            return BSG_ERR_NO_PLAN;
    } else {
        // 128-wide tiles while they number at most 4 per SM; beyond that,
        // NVFP4 slices go to the CTA pair's 256-row tile rows (up to its
        // slice bound; on the 64-expert MoE workload 8 % faster than the
        // 1-SM 128 x 256 tiles, which give a slice of 129..256 rows a
        // second tile row that streams its weights again), else 256-wide
        // 1-SM tiles
        const long long tiles128 = mt_bound * (long long)((N + 127) / 128);
        const bool few = tiles128 <= 4LL * ds->sms;
        if (!dense && !few && N > 128 && E <= bsg::kPairMaxGroups) {
            plan = bsg::find_plan("nvfp4_tc2_256x256_s5_acc1");
            if (plan >= 0)
                return run_grouped_pair(plan, E, M, N, K, A, sfa, B, sfb, offs, alpha, epi, D, stream, ds);
        }
        plan = bsg::find_plan(dense ? (few ? "nvfp4bf16_tc1_128x128_s8_acc2_tmema" : "nvfp4bf16_tc1_128x256_s5_acc1_tmema")
                                    : (few ? "nvfp4_tc1_128x128_s5_acc2" : "nvfp4_tc1_128x256_s3_acc1"));
        if (plan < 0)
            return BSG_ERR_NO_PLAN;
    }
    const PlanInfo &pi = bsg::plan_info(plan);
    const uint64_t row_bytes = (uint64_t)K / 2u;
    const uint64_t b_row_bytes = dense ? 2u * (uint64_t)K : row_bytes;
    GemmMaps maps;
    std::memset(&maps, 0, sizeof maps);
    int rc;
    // dense: A's codes unswizzled, 32 bytes a row per 64-K stage (expanded
    // on the GPU); B 16-bit, 128 bytes a row per stage
    if ((rc = encode_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, row_bytes, (uint64_t)M, row_bytes,
                        dense ? 32 : 128, 128,
                        dense ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B)) != BSG_OK ||
        (rc = encode_2d(&maps.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, b_row_bytes, (uint64_t)E * (uint64_t)N,
                        b_row_bytes, 128, (uint32_t)pi.bn)) != BSG_OK ||
        (rc = encode_2d(&maps.d, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, (uint64_t)N, d_rows(M, epi),
                        (uint64_t)N * 2u, 64, 32)) != BSG_OK)
        return rc;
    maps.sfa = maps.a;
    maps.sfb = maps.a;
    GemmArgs a;
    std::memset(&a, 0, sizeof a);
    a.M = M;
    a.N = N;
    a.K = K;
    a.num_m_tiles = (int)mt_bound;      // bound only: the kernel counts the slices' tile rows
    a.num_n_tiles = (N + pi.bn - 1) / pi.bn;
    a.num_k_blocks = K / pi.k_block;
    a.raster_group = g_raster_group.load();
    a.sf_col_blocks = (K / 16 + 3) / 4;
    a.sfb_row_blocks = (N + 127) / 128;
    a.sfa = sfa;
    a.sfb = sfb;
    a.alpha = alpha;
    a.status = ds->status;
    a.timeout_ns = g_watchdog_ns.load();
    set_epilogue(a, epi, D);
    a.num_groups = E;
    a.group_offs = offs;
    a.sfb_group_bytes = dense ? 0 : swizzled_bytes(N, K);
    a.b_f16 = b_f16 ? 1 : 0;
    a.pdl = g_pdl.load();
    const long long ctas = mt_bound * a.num_n_tiles;
    const int resident = bsg::max_resident_ctas(plan, ds->sms);
    if (resident < 1)
        return BSG_ERR_CUDA;
    const int grid = (int)(ctas < resident ? ctas : resident);
    if (bsg::launch_gemm(plan, maps, a, grid, stream) != cudaSuccess)
        return BSG_ERR_CUDA;
    ++t_last_launches;
    t_last_plan = pi.name;
    return BSG_OK;
}

// K-ragged (inner-expert) NVFP4 x dense GEMM: koffs splits K into E slices
// and slice e writes rows [e*M, e*M + M) of D. Tiles: E x M/128 x N/BN.
int run_kgrouped(int E, int M, int N, int K, const void *A, const uint8_t *sfa, const void *B, const int32_t *koffs,
                 float alpha, const Epilogue &epi, void *D, cudaStream_t stream, DeviceState *ds, bool b_f16)
{
    const long long m_tiles = (M + 127) / 128;
    int plan;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        plan = g_forced_plan;
    }
    if (plan >= 0) {
        if (!grouped_dense_plan(bsg::plan_info(plan)))
            return BSG_ERR_NO_PLAN;
    } else {
        const long long tiles128 = (long long)E * m_tiles * (long long)((N + 127) / 128);
        plan = bsg::find_plan(tiles128 <= 4LL * ds->sms ? "nvfp4bf16_tc1_128x128_s8_acc2_tmema"
                                                       : "nvfp4bf16_tc1_128x256_s5_acc1_tmema");
        if (plan < 0)
            return BSG_ERR_NO_PLAN;
    }
    const PlanInfo &pi = bsg::plan_info(plan);
    const uint64_t row_bytes = (uint64_t)K / 2u;
    GemmMaps maps;
    std::memset(&maps, 0, sizeof maps);
    int rc;
    if ((rc = encode_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, A, row_bytes, (uint64_t)M, row_bytes, 32, 128,
                        CU_TENSOR_MAP_SWIZZLE_NONE)) != BSG_OK ||
        (rc = encode_2d(&maps.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, B, 2u * (uint64_t)K, (uint64_t)N,
                        2u * (uint64_t)K, 128, (uint32_t)pi.bn)) != BSG_OK ||
        (rc = encode_2d(&maps.d, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, (uint64_t)N, (uint64_t)E * (uint64_t)M,
                        (uint64_t)N * 2u, 64, 32)) != BSG_OK)
        return rc;
    maps.sfa = maps.a;
    maps.sfb = maps.a;
    GemmArgs a;
    std::memset(&a, 0, sizeof a);
    a.M = M;
    a.N = N;
    a.K = K;
    a.num_m_tiles = (int)m_tiles;
    a.num_n_tiles = (N + pi.bn - 1) / pi.bn;
    a.num_k_blocks = K / pi.k_block;
    a.raster_group = g_raster_group.load();
    a.sf_col_blocks = (K / 16 + 3) / 4;
    a.sfa = sfa;
    a.alpha = alpha;
    a.status = ds->status;
    a.timeout_ns = g_watchdog_ns.load();
    set_epilogue(a, epi, D);
    a.num_groups = E;
    a.group_offs = koffs;
    a.k_grouped = 1;
    a.b_f16 = b_f16 ? 1 : 0;
    a.pdl = g_pdl.load();
    const long long ctas = (long long)E * m_tiles * a.num_n_tiles;
    const int resident = bsg::max_resident_ctas(plan, ds->sms);
    if (resident < 1)
        return BSG_ERR_CUDA;
    const int grid = (int)(ctas < resident ? ctas : resident);
    if (bsg::launch_gemm(plan, maps, a, grid, stream) != cudaSuccess)
        return BSG_ERR_CUDA;
    ++t_last_launches;
    t_last_plan = pi.name;
    return BSG_OK;
}

// Both operands' scales of one GEMM: one launch while the two grids' block
// rows fit the grid's y limit, else one launch each.
cudaError_t swizzle_both(int M, int N, int K, const uint8_t *sfa, uint8_t *out_a, const uint8_t *sfb,
                         uint8_t *out_b, cudaStream_t s, int *launches)
{
    if ((long long)(M + 127) / 128 + (N + 127) / 128 <= 65535) {
        *launches = 1;
        return bsg::launch_swizzle_scales2(M, N, K, sfa, out_a, sfb, out_b, s);
    }
    *launches = 2;
    cudaError_t e = bsg::launch_swizzle_scales(M, K, sfa, out_a, s);
    return e != cudaSuccess ? e : bsg::launch_swizzle_scales(N, K, sfb, out_b, s);
}

int check_nvfp4_args(int M, int N, int K, const void *A, const void *sfA, const void *B,
                     const void *sfB, void *D)
{
    if (!A || !sfA || !B || !sfB || !D)
        return BSG_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 256 || (K % 256) != 0 || (N % 8) != 0)
        return BSG_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(sfA) || !aligned16(B) || !aligned16(sfB) || !aligned16(D))
        return BSG_ERR_MISALIGNED;
    return BSG_OK;
}

int check_fp8_args(int M, int N, int K, const void *A, const float *sA, const void *B, const float *sB,
                   void *D)
{
    if (!A || !B || !D)
        return BSG_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 128 || (K % 128) != 0 || (N % 8) != 0)
        return BSG_ERR_INVALID_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(D) ||
        (sA && (reinterpret_cast<uintptr_t>(sA) & 3u)) || (sB && (reinterpret_cast<uintptr_t>(sB) & 3u)))
        return BSG_ERR_MISALIGNED;
    return BSG_OK;
}

// bias 16-byte aligned (read as float4), gamma and scatter 4-byte aligned;
// m_out == M without scatter, >= 1 with it.
int check_epilogue_args(int M, const float *bias, const float *gamma, const int32_t *scatter, int m_out)
{
    if (scatter ? m_out < 1 : m_out != M)
        return BSG_ERR_INVALID_ARG;
    if ((bias && !aligned16(bias)) || (gamma && (reinterpret_cast<uintptr_t>(gamma) & 3u)) ||
        (scatter && (reinterpret_cast<uintptr_t>(scatter) & 3u)))
        return BSG_ERR_MISALIGNED;
    return BSG_OK;
}

// Grow the workspace of the current device (caller holds no lock).
int ensure_workspace(DeviceState *ds, size_t bytes)
{
    std::lock_guard<std::mutex> lk(g_mu);
    if (ds->ws_bytes >= bytes)
        return BSG_OK;
    if (ds->ws) {
        cudaFree(ds->ws);   // synchronises the device: no pending work still reads it
        ds->ws = nullptr;
        ds->ws_bytes = 0;
    }
    if (cudaMalloc(reinterpret_cast<void **>(&ds->ws), bytes) != cudaSuccess) {
        cudaGetLastError();
        ds->ws = nullptr;
        return BSG_ERR_OUT_OF_MEMORY;
    }
    ds->ws_bytes = bytes;
    return BSG_OK;
}

size_t round256(size_t x) { return (x + 255u) & ~(size_t)255u; }

}  // namespace

namespace bsg {
int num_plans() { return tc1_num_plans() + pair_num_plans() + skinny_num_plans(); }

const PlanInfo &plan_info(int id)
{
    if (id < tc1_num_plans())
        return tc1_plan(id);
    id -= tc1_num_plans();
    return id < pair_num_plans() ? pair_plan(id) : skinny_plan(id - pair_num_plans());
}

cudaError_t launch_gemm(int id, const GemmMaps &maps, const GemmArgs &args, int grid,
                        cudaStream_t stream)
{
    if (id < tc1_num_plans())
        return tc1_launch(id, maps, args, grid, stream);
    return pair_launch(id - tc1_num_plans(), maps, args, grid, stream);
}

cudaError_t set_max_dynamic_smem(const void *kern, int bytes)
{
    struct Done {
        int dev;
        const void *kern;
        int bytes;
    };
    static std::vector<Done> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lk(g_mu);
    for (const Done &d : done)
        if (d.dev == dev && d.kern == kern && d.bytes == bytes)
            return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
        done.push_back(Done{dev, kern, bytes});
    return e;
}

int max_resident_ctas(int id, int num_sms)
{
    if (id < tc1_num_plans())
        return num_sms;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return 0;
    static int cache[kMaxDevices][16] = {};
    const int j = id - tc1_num_plans();
    if (j >= 16)
        return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (cache[dev][j] == 0)
        cache[dev][j] = 2 * pair_max_clusters(j);
    return cache[dev][j];
}

int validate_nvfp4_call(int M, int N, int K, const void *A, const void *sfA, const void *B, const void *sfB,
                        void *D)
{
    t_last_launches = 0;
    int rc = check_nvfp4_args(M, N, K, A, sfA, B, sfB, D);
    if (rc != BSG_OK)
        return rc;
    DeviceState *ds = nullptr;
    return current_device(&ds);
}

void add_launches(int n) { t_last_launches += n; }

int find_plan(const char *name)
{
    if (!name)
        return -1;
    for (int i = 0; i < num_plans(); ++i)
        if (std::strcmp(plan_info(i).name, name) == 0)
            return i;
    return -1;
}
}  // namespace bsg

extern "C" {

int nvfp4_gemm_swizzled(int M, int N, int K, const void *A, const void *sfA_swz, const void *B,
                        const void *sfB_swz, float alpha, void *D, bsg_stream_t stream)
{
    t_last_launches = 0;
    int rc = check_nvfp4_args(M, N, K, A, sfA_swz, B, sfB_swz, D);
    if (rc != BSG_OK)
        return rc;
    DeviceState *ds = nullptr;
    if ((rc = current_device(&ds)) != BSG_OK)
        return rc;
    return run_gemm(Kind::NVFP4, M, N, K, A, B, static_cast<const uint8_t *>(sfA_swz),
                    static_cast<const uint8_t *>(sfB_swz), nullptr, nullptr, alpha, D,
                    reinterpret_cast<cudaStream_t>(stream), ds);
}

int nvfp4_gemm(int M, int N, int K, const void *A, const void *sfA, const void *B, const void *sfB,
               float alpha, void *D, bsg_stream_t stream)
{
    t_last_launches = 0;
    int rc = check_nvfp4_args(M, N, K, A, sfA, B, sfB, D);
    if (rc != BSG_OK)
        return rc;
    DeviceState *ds = nullptr;
    if ((rc = current_device(&ds)) != BSG_OK)
        return rc;
    const size_t bytes_a = round256(swizzled_bytes(M, K));
    const size_t bytes_b = round256(swizzled_bytes(N, K));
    if ((rc = ensure_workspace(ds, bytes_a + bytes_b)) != BSG_OK)
        return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint8_t *swz_a = ds->ws;
    uint8_t *swz_b = ds->ws + bytes_a;
    int swz_launches = 0;
    if (swizzle_both(M, N, K, static_cast<const uint8_t *>(sfA), swz_a, static_cast<const uint8_t *>(sfB), swz_b, s,
                     &swz_launches) != cudaSuccess)
        return BSG_ERR_CUDA;
    t_last_launches = swz_launches;
    return run_gemm(Kind::NVFP4, M, N, K, A, B, swz_a, swz_b, nullptr, nullptr, alpha, D, s, ds);
}

int nvfp4_swizzle_scales2(int M, int N, int K, const void *sfA, void *sfA_swz, const void *sfB, void *sfB_swz,
                          bsg_stream_t stream)
{
    t_last_launches = 0;
    if (!sfA || !sfA_swz || !sfB || !sfB_swz || M < 1 || N < 1 || K < 16 || (K % 16) != 0)
        return BSG_ERR_INVALID_ARG;
    if (!aligned16(sfA_swz) || !aligned16(sfB_swz))
        return BSG_ERR_MISALIGNED;
    DeviceState *ds = nullptr;
    int rc = current_device(&ds);
    if (rc != BSG_OK)
        return rc;
    int n = 0;
    if (swizzle_both(M, N, K, static_cast<const uint8_t *>(sfA), static_cast<uint8_t *>(sfA_swz),
                     static_cast<const uint8_t *>(sfB), static_cast<uint8_t *>(sfB_swz),
                     reinterpret_cast<cudaStream_t>(stream), &n) != cudaSuccess)
        return BSG_ERR_CUDA;
    t_last_launches = n;
    return BSG_OK;
}

size_t nvfp4_packed_operand_bytes(int rows, int K)
{
    if (rows < 1 || K < 256 || (K % 256) != 0)
        return 0;
    return (size_t)((rows + 127) / 128) * 128u * (size_t)(K / 2);
}

int nvfp4_pack_operand(int rows, int K, const void *X, void *out, bsg_stream_t stream)
{
    t_last_launches = 0;
    if (!X || !out || rows < 1 || K < 256 || (K % 256) != 0 || (rows + 127) / 128 > 65535)
        return BSG_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(out))
        return BSG_ERR_MISALIGNED;
    DeviceState *ds = nullptr;
    int rc = current_device(&ds);
    if (rc != BSG_OK)
        return rc;
    if (bsg::launch_pack_operand(rows, K, static_cast<const uint8_t *>(X), static_cast<uint8_t *>(out),
                                 reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return BSG_ERR_CUDA;
    t_last_launches = 1;
    return BSG_OK;
}

int nvfp4_gemm_packed_ex(int M, int N, int K, const void *A_packed, const void *sfA_swz, const void *B_packed,
                         const void *sfB_swz, float alpha, const float *bias, const float *gamma,
                         const int32_t *scatter, int m_out, void *D, bsg_stream_t stream)
{
    t_last_launches = 0;
    int rc = check_nvfp4_args(M, N, K, A_packed, sfA_swz, B_packed, sfB_swz, D);
    if (rc != BSG_OK || (rc = check_epilogue_args(M, bias, gamma, scatter, m_out)) != BSG_OK)
        return rc;
    DeviceState *ds = nullptr;
    if ((rc = current_device(&ds)) != BSG_OK)
        return rc;
    Epilogue e;
    e.bias = bias;
    e.gamma = gamma;
    e.scatter = scatter;
    e.m_out = m_out;
    return run_gemm(Kind::NVFP4, M, N, K, nullptr, nullptr, static_cast<const uint8_t *>(sfA_swz),
                    static_cast<const uint8_t *>(sfB_swz), nullptr, nullptr, alpha, D,
                    reinterpret_cast<cudaStream_t>(stream), ds, e, false, static_cast<const uint8_t *>(A_packed),
                    static_cast<const uint8_t *>(B_packed));
}

int nvfp4_gemm_packed(int M, int N, int K, const void *A_packed, const void *sfA_swz, const void *B_packed,
                      const void *sfB_swz, float alpha, void *D, bsg_stream_t stream)
{
    return nvfp4_gemm_packed_ex(M, N, K, A_packed, sfA_swz, B_packed, sfB_swz, alpha, nullptr, nullptr, nullptr, M,
                                D, stream);
}

static int quantize(bool tiles, int rows, int K, const void *X, void *packed, void *sf_swz, void *sf_rowmajor,
                    float *global, bsg_stream_t stream)
{
    t_last_launches = 0;
    if (!X || !packed || !sf_swz || !global || rows < 1 || K < 16 || (K % 16) != 0)
        return BSG_ERR_INVALID_ARG;
    if (tiles && (K % 256) != 0)
        return BSG_ERR_INVALID_ARG;
    if (!aligned16(X) || !aligned16(packed) || !aligned16(sf_swz) ||
        (reinterpret_cast<uintptr_t>(global) & 7u) != 0)
        return BSG_ERR_MISALIGNED;
    DeviceState *ds = nullptr;
    int rc = current_device(&ds);
    if (rc != BSG_OK)
        return rc;
    if (bsg::launch_nvfp4_quantize(rows, K, X, static_cast<uint8_t *>(packed), static_cast<uint8_t *>(sf_swz),
                                   static_cast<uint8_t *>(sf_rowmajor), global, ds->sms,
                                   reinterpret_cast<cudaStream_t>(stream), tiles) != cudaSuccess)
        return BSG_ERR_CUDA;
    t_last_launches = 2;
    return BSG_OK;
}

int nvfp4_quantize(int rows, int K, const void *X, void *packed, void *sf_swz, void *sf_rowmajor,
                   float *global, bsg_stream_t stream)
{
    return quantize(false, rows, K, X, packed, sf_swz, sf_rowmajor, global, stream);
}

int nvfp4_quantize_tiles(int rows, int K, const void *X, void *packed_tiles, void *sf_swz, void *sf_rowmajor,
                         float *global, bsg_stream_t stream)
{
    return quantize(true, rows, K, X, packed_tiles, sf_swz, sf_rowmajor, global, stream);
}

int nvfp4_swizzle_scales(int rows, int K, const void *sf, void *sf_swz, bsg_stream_t stream)
{
    t_last_launches = 0;
    if (!sf || !sf_swz || rows < 1 || K < 16 || (K % 16) != 0)
        return BSG_ERR_INVALID_ARG;
    if (!aligned16(sf_swz))
        return BSG_ERR_MISALIGNED;
    DeviceState *ds = nullptr;
    int rc = current_device(&ds);
    if (rc != BSG_OK)
        return rc;
    if (bsg::launch_swizzle_scales(rows, K, static_cast<const uint8_t *>(sf),
                                   static_cast<uint8_t *>(sf_swz),
                                   reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return BSG_ERR_CUDA;
    t_last_launches = 1;
    return BSG_OK;
}

size_t nvfp4_swizzled_scale_bytes(int rows, int K) { return swizzled_bytes(rows, K); }

int fp8_gemm(int M, int N, int K, const void *A, const float *sA, const void *B, const float *sB,
             float alpha, void *D, bsg_stream_t stream)
{
    t_last_launches = 0;
    int rc = check_fp8_args(M, N, K, A, sA, B, sB, D);
    if (rc != BSG_OK)
        return rc;
    DeviceState *ds = nullptr;
    rc = current_device(&ds);
    if (rc != BSG_OK)
        return rc;
    return run_gemm(Kind::FP8, M, N, K, A, B, nullptr, nullptr, sA, sB, alpha, D,
                    reinterpret_cast<cudaStream_t>(stream), ds);
}

int nvfp4_gemm_ex(int M, int N, int K, const void *A, const void *sfA_swz, const void *B,
                  const void *sfB_swz, float alpha, const float *bias, const float *gamma,
                  const int32_t *scatter, int m_out, void *D, bsg_stream_t stream)
{
    t_last_launches = 0;
    int rc = check_nvfp4_args(M, N, K, A, sfA_swz, B, sfB_swz, D);
    if (rc != BSG_OK || (rc = check_epilogue_args(M, bias, gamma, scatter, m_out)) != BSG_OK)
        return rc;
    DeviceState *ds = nullptr;
    if ((rc = current_device(&ds)) != BSG_OK)
        return rc;
    Epilogue e;
    e.bias = bias;
    e.gamma = gamma;
    e.scatter = scatter;
    e.m_out = m_out;
    return run_gemm(Kind::NVFP4, M, N, K, A, B, static_cast<const uint8_t *>(sfA_swz),
                    static_cast<const uint8_t *>(sfB_swz), nullptr, nullptr, alpha, D,
                    reinterpret_cast<cudaStream_t>(stream), ds, e);
}

int fp8_gemm_ex(int M, int N, int K, const void *A, const float *sA, const void *B, const float *sB,
                float alpha, const float *bias, const float *gamma, const int32_t *scatter, int m_out,
                void *D, bsg_stream_t stream)
{
    t_last_launches = 0;
    int rc = check_fp8_args(M, N, K, A, sA, B, sB, D);
    if (rc != BSG_OK || (rc = check_epilogue_args(M, bias, gamma, scatter, m_out)) != BSG_OK)
        return rc;
    DeviceState *ds = nullptr;
    if ((rc = current_device(&ds)) != BSG_OK)
        return rc;
    Epilogue e;
    e.bias = bias;
    e.gamma = gamma;
    e.scatter = scatter;
    e.m_out = m_out;
    return run_gemm(Kind::FP8, M, N, K, A, B, nullptr, nullptr, sA, sB, alpha, D,
                    reinterpret_cast<cudaStream_t>(stream), ds, e);
}

size_t nvfp4_grouped_scale_bytes(int E, int M, int K)
{
    if (E < 1 || E > bsg::kMaxGroups || M < 0 || K < 16 || (K % 16) != 0)
        return 0;
    return ((size_t)(M + 127) / 128u + (size_t)E) * 128u * ((size_t)(K / 16 + 3) / 4u * 4u);
}

int nvfp4_swizzle_scales_grouped(int E, int M, int K, const int32_t *offs, const void *sf, void *sf_swz,
                                 bsg_stream_t stream)
{
    t_last_launches = 0;
    if (!offs || !sf || !sf_swz || E < 1 || E > bsg::kMaxGroups || M < 1 || K < 16 || (K % 16) != 0)
        return BSG_ERR_INVALID_ARG;
    if (!aligned16(sf_swz) || (reinterpret_cast<uintptr_t>(offs) & 3u))
        return BSG_ERR_MISALIGNED;
    DeviceState *ds = nullptr;
    int rc = current_device(&ds);
    if (rc != BSG_OK)
        return rc;
    if (bsg::launch_swizzle_scales_grouped(E, M, K, offs, static_cast<const uint8_t *>(sf),
                                           static_cast<uint8_t *>(sf_swz),
                                           reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return BSG_ERR_CUDA;
    t_last_launches = 1;
    return BSG_OK;
}

int nvfp4_grouped_gemm(int E, int M, int N, int K, const void *A, const void *sfA_swz, const void *B,
                       const void *sfB_swz, const int32_t *offs, float alpha, const float *bias,
                       const float *gamma, const int32_t *scatter, int m_out, void *D, bsg_stream_t stream)
{
    t_last_launches = 0;
    if (!offs || E < 1 || E > bsg::kMaxGroups)
        return BSG_ERR_INVALID_ARG;
    int rc = check_nvfp4_args(M, N, K, A, sfA_swz, B, sfB_swz, D);
    if (rc != BSG_OK || (rc = check_epilogue_args(M, bias, gamma, scatter, m_out)) != BSG_OK)
        return rc;
    if (reinterpret_cast<uintptr_t>(offs) & 3u)
        return BSG_ERR_MISALIGNED;
    DeviceState *ds = nullptr;
    if ((rc = current_device(&ds)) != BSG_OK)
        return rc;
    Epilogue e;
    e.bias = bias;
    e.gamma = gamma;
    e.scatter = scatter;
    e.m_out = m_out;
    return run_grouped(E, M, N, K, A, static_cast<const uint8_t *>(sfA_swz), B,
                       static_cast<const uint8_t *>(sfB_swz), offs, alpha, e, D,
                       reinterpret_cast<cudaStream_t>(stream), ds);
}

static int dense_gemm(bool b_f16, int M, int N, int K, const void *A, const void *sfA_swz, const void *B,
                      float alpha, const float *bias, const float *gamma, const int32_t *scatter, int m_out,
                      void *D, bsg_stream_t stream)
{
    t_last_launches = 0;
    if (!A || !sfA_swz || !B || !D)
        return BSG_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 64 || (K % 64) != 0 || (N % 8) != 0)
        return BSG_ERR_INVALID_ARG;
    int rc = check_epilogue_args(M, bias, gamma, scatter, m_out);
    if (rc != BSG_OK)
        return rc;
    if (!aligned16(A) || !aligned16(sfA_swz) || !aligned16(B) || !aligned16(D))
        return BSG_ERR_MISALIGNED;
    DeviceState *ds = nullptr;
    if ((rc = current_device(&ds)) != BSG_OK)
        return rc;
    Epilogue e;
    e.bias = bias;
    e.gamma = gamma;
    e.scatter = scatter;
    e.m_out = m_out;
    return run_gemm(Kind::NVFP4_BF16, M, N, K, A, B, static_cast<const uint8_t *>(sfA_swz), nullptr, nullptr,
                    nullptr, alpha, D, reinterpret_cast<cudaStream_t>(stream), ds, e, b_f16);
}

int nvfp4_dense_gemm(int M, int N, int K, const void *A, const void *sfA_swz, const void *B, float alpha,
                     const float *bias, const float *gamma, const int32_t *scatter, int m_out, void *D,
                     bsg_stream_t stream)
{
    return dense_gemm(false, M, N, K, A, sfA_swz, B, alpha, bias, gamma, scatter, m_out, D, stream);
}

int nvfp4_dense_f16_gemm(int M, int N, int K, const void *A, const void *sfA_swz, const void *B, float alpha,
                         const float *bias, const float *gamma, const int32_t *scatter, int m_out, void *D,
                         bsg_stream_t stream)
{
    return dense_gemm(true, M, N, K, A, sfA_swz, B, alpha, bias, gamma, scatter, m_out, D, stream);
}

static int dense_grouped_gemm(bool b_f16, int E, int M, int N, int K, const void *A, const void *sfA_swz,
                              const void *B, const int32_t *offs, float alpha, const float *bias,
                              const float *gamma, const int32_t *scatter, int m_out, void *D, bsg_stream_t stream)
{
    t_last_launches = 0;
    if (!A || !sfA_swz || !B || !D || !offs || E < 1 || E > bsg::kMaxGroups)
        return BSG_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 64 || (K % 64) != 0 || (N % 8) != 0)
        return BSG_ERR_INVALID_ARG;
    int rc = check_epilogue_args(M, bias, gamma, scatter, m_out);
    if (rc != BSG_OK)
        return rc;
    if (!aligned16(A) || !aligned16(sfA_swz) || !aligned16(B) || !aligned16(D) ||
        (reinterpret_cast<uintptr_t>(offs) & 3u))
        return BSG_ERR_MISALIGNED;
    DeviceState *ds = nullptr;
    if ((rc = current_device(&ds)) != BSG_OK)
        return rc;
    Epilogue e;
    e.bias = bias;
    e.gamma = gamma;
    e.scatter = scatter;
    e.m_out = m_out;
    return run_grouped(E, M, N, K, A, static_cast<const uint8_t *>(sfA_swz), B, nullptr, offs, alpha, e, D,
                       reinterpret_cast<cudaStream_t>(stream), ds, true, b_f16);
}

static int dense_kgrouped_gemm(bool b_f16, int E, int M, int N, int K, const void *A, const void *sfA_swz,
                               const void *B, const int32_t *koffs, float alpha, const float *bias,
                               const float *gamma, void *D, bsg_stream_t stream)
{
    t_last_launches = 0;
    if (!A || !sfA_swz || !B || !D || !koffs || E < 1 || E > bsg::kMaxGroups)
        return BSG_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 64 || (K % 64) != 0 || (N % 8) != 0)
        return BSG_ERR_INVALID_ARG;
    int rc = check_epilogue_args(M, bias, gamma, nullptr, M);
    if (rc != BSG_OK)
        return rc;
    if (!aligned16(A) || !aligned16(sfA_swz) || !aligned16(B) || !aligned16(D) ||
        (reinterpret_cast<uintptr_t>(koffs) & 3u))
        return BSG_ERR_MISALIGNED;
    DeviceState *ds = nullptr;
    if ((rc = current_device(&ds)) != BSG_OK)
        return rc;
    Epilogue e;
    e.bias = bias;
    e.gamma = gamma;
    e.m_out = M;
    return run_kgrouped(E, M, N, K, A, static_cast<const uint8_t *>(sfA_swz), B, koffs, alpha, e, D,
                        reinterpret_cast<cudaStream_t>(stream), ds, b_f16);
}

int nvfp4_dense_kgrouped_gemm(int E, int M, int N, int K, const void *A, const void *sfA_swz, const void *B,
                              const int32_t *koffs, float alpha, const float *bias, const float *gamma, void *D,
                              bsg_stream_t stream)
{
    return dense_kgrouped_gemm(false, E, M, N, K, A, sfA_swz, B, koffs, alpha, bias, gamma, D, stream);
}

int nvfp4_dense_f16_kgrouped_gemm(int E, int M, int N, int K, const void *A, const void *sfA_swz, const void *B,
                                  const int32_t *koffs, float alpha, const float *bias, const float *gamma, void *D,
                                  bsg_stream_t stream)
{
    return dense_kgrouped_gemm(true, E, M, N, K, A, sfA_swz, B, koffs, alpha, bias, gamma, D, stream);
}

int nvfp4_dense_grouped_gemm(int E, int M, int N, int K, const void *A, const void *sfA_swz, const void *B,
                             const int32_t *offs, float alpha, const float *bias, const float *gamma,
                             const int32_t *scatter, int m_out, void *D, bsg_stream_t stream)
{
    return dense_grouped_gemm(false, E, M, N, K, A, sfA_swz, B, offs, alpha, bias, gamma, scatter, m_out, D,
                              stream);
}

int nvfp4_dense_f16_grouped_gemm(int E, int M, int N, int K, const void *A, const void *sfA_swz, const void *B,
                                 const int32_t *offs, float alpha, const float *bias, const float *gamma,
                                 const int32_t *scatter, int m_out, void *D, bsg_stream_t stream)
{
    return dense_grouped_gemm(true, E, M, N, K, A, sfA_swz, B, offs, alpha, bias, gamma, scatter, m_out, D,
                              stream);
}

int bsg_reserve_workspace(int device, size_t bytes)
{
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(device) != cudaSuccess)
        return BSG_ERR_CUDA;
    DeviceState *ds = nullptr;
    int rc = current_device(&ds);
    if (rc == BSG_OK)
        rc = ensure_workspace(ds, bytes);
    cudaSetDevice(prev);
    return rc;
}

int bsg_get_device_status(bsg_stream_t stream)
{
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    DeviceState *ds = nullptr;
    int rc = current_device(&ds);
    if (rc != BSG_OK)
        return rc;
    unsigned int v = 0;
    if (cudaMemcpy(&v, ds->status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(ds->status, 0, sizeof v) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
        return BSG_ERR_CUDA;
    t_last_status_word = v;
    if (e != cudaSuccess)
        return BSG_ERR_CUDA;
    return v ? BSG_ERR_DEVICE_TIMEOUT : BSG_OK;
}

uint32_t bsg_last_status_word(void) { return t_last_status_word; }

int bsg_set_watchdog_ns(uint64_t ns)
{
    g_watchdog_ns.store(ns ? (unsigned long long)ns : kDefaultWatchdogNs);
    return BSG_OK;
}

int bsg_set_pdl(int on)
{
    if (on < 0 || on > 2)
        return BSG_ERR_INVALID_ARG;
    g_pdl.store(on);
    return BSG_OK;
}

int bsg_set_raster_group(int m_tiles)
{
    if (m_tiles < 0 || m_tiles > 1024)
        return BSG_ERR_INVALID_ARG;
    g_raster_group.store(m_tiles == 0 ? kDefaultRasterGroup : m_tiles);
    return BSG_OK;
}

int bsg_set_skinny_splits(int splits)
{
    if (splits < 0 || splits > 8 || splits == 7)
        return BSG_ERR_INVALID_ARG;
    g_skinny_splits.store(splits);
    return BSG_OK;
}

int bsg_watchdog_selftest(uint64_t ns, bsg_stream_t stream)
{
    if (ns == 0)
        return BSG_ERR_INVALID_ARG;
    DeviceState *ds = nullptr;
    int rc = current_device(&ds);
    if (rc != BSG_OK)
        return rc;
    if (bsg::launch_watchdog_probe(ds->status, (unsigned long long)ns,
                                   reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return BSG_ERR_CUDA;
    return BSG_OK;
}

int bsg_measure_ingress(size_t src_bytes, int stages, int tensor_boxes, double *bytes_per_cycle_per_sm,
                        double *total_gbs)
{
    // tensor boxes: rows of 8192 bytes (an NVFP4 operand row at K = 16384),
    // at least two 128-row tile rows of them
    const size_t pitch = 8192;
    if (!bytes_per_cycle_per_sm || stages < 1 || stages > bsg::probe_max_stages() ||
        src_bytes < (size_t)4 * (size_t)bsg::probe_slot_bytes() || (tensor_boxes && src_bytes < 256 * pitch))
        return BSG_ERR_INVALID_ARG;
    DeviceState *ds = nullptr;
    int rc = current_device(&ds);
    if (rc != BSG_OK)
        return rc;
    const int iters = 4000;
    uint8_t *src = nullptr;
    unsigned long long *cyc = nullptr;
    cudaStream_t st = nullptr;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    float ms = 0.0f;
    rc = BSG_ERR_CUDA;
    CUtensorMap tm;
    std::memset(&tm, 0, sizeof tm);
    const size_t rows = (src_bytes / pitch) / 128 * 128;
    auto launch = [&]() {
        if (!tensor_boxes)
            return bsg::launch_ingress_probe(src, src_bytes, stages, iters, ds->sms, ds->status, g_watchdog_ns.load(),
                                             cyc, st);
        return bsg::launch_tma_ingress_probe(tm, (int)(pitch / 128), (int)(rows / 128), stages, iters, ds->sms,
                                             ds->status, g_watchdog_ns.load(), cyc, st);
    };
    if (cudaMalloc(&src, src_bytes) == cudaSuccess && cudaMalloc(&cyc, sizeof(unsigned long long) * ds->sms) == cudaSuccess &&
        cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) == cudaSuccess && cudaEventCreate(&e0) == cudaSuccess &&
        cudaEventCreate(&e1) == cudaSuccess && cudaMemsetAsync(src, 0x5A, src_bytes, st) == cudaSuccess &&
        (!tensor_boxes || encode_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, src, pitch, rows, pitch, 128, 128) == BSG_OK) &&
        // one untimed pass (first touch of the source), then the timed one
        launch() == cudaSuccess && cudaEventRecord(e0, st) == cudaSuccess && launch() == cudaSuccess &&
        cudaEventRecord(e1, st) == cudaSuccess && cudaStreamSynchronize(st) == cudaSuccess &&
        cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess) {
        std::vector<unsigned long long> c((size_t)ds->sms);
        unsigned int word = 0;
        if (cudaMemcpy(c.data(), cyc, sizeof(unsigned long long) * ds->sms, cudaMemcpyDeviceToHost) == cudaSuccess &&
            cudaMemcpy(&word, ds->status, sizeof word, cudaMemcpyDeviceToHost) == cudaSuccess) {
            if (word != 0) {
                rc = BSG_ERR_DEVICE_TIMEOUT;
            } else {
                double mean = 0.0;
                for (unsigned long long v : c)
                    mean += (double)v;
                mean /= (double)ds->sms;
                const double per_cta = (double)iters * (double)bsg::probe_slot_bytes();
                *bytes_per_cycle_per_sm = mean > 0.0 ? per_cta / mean : 0.0;
                if (total_gbs)
                    *total_gbs = ms > 0.0f ? per_cta * ds->sms / ((double)ms * 1e-3) / 1e9 : 0.0;
                rc = BSG_OK;
            }
        }
    }
    if (e0)
        cudaEventDestroy(e0);
    if (e1)
        cudaEventDestroy(e1);
    if (st)
        cudaStreamDestroy(st);
    cudaFree(src);
    cudaFree(cyc);
    return rc;
}

int bsg_force_plan(const char *name)
{
    int id = -1;
    if (name && name[0]) {
        id = bsg::find_plan(name);
        if (id < 0)
            return BSG_ERR_NO_PLAN;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    g_forced_plan = id;
    return BSG_OK;
}

int bsg_select_plan(int kind, int M, int N, int K, int num_sms, char *name, size_t name_len)
{
    if (kind < 0 || kind > 2 || M < 1 || N < 1 || K < 1 || num_sms < 1 || !name || name_len == 0)
        return BSG_ERR_INVALID_ARG;
    int plan = -1;
    int rc = choose_plan(static_cast<Kind>(kind), M, N, K, num_sms, &plan);
    if (rc != BSG_OK)
        return rc;
    std::strncpy(name, bsg::plan_info(plan).name, name_len - 1);
    name[name_len - 1] = '\0';
    return BSG_OK;
}

int bsg_last_launch_count(void) { return t_last_launches; }

const char *bsg_last_plan_name(void) { return t_last_plan; }

const char *bsg_error_string(int code)
{
    switch (code) {
    case BSG_OK: return "ok";
    case BSG_ERR_INVALID_ARG: return "invalid argument";
    case BSG_ERR_MISALIGNED: return "misaligned pointer (16-byte alignment required)";
    case BSG_ERR_UNSUPPORTED_DEVICE: return "unsupported device (compute capability 10.3 required)";
    case BSG_ERR_NO_PLAN: return "no kernel plan for this request";
    case BSG_ERR_CUDA: return "CUDA error";
    case BSG_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case BSG_ERR_OUT_OF_MEMORY: return "workspace allocation failed";
    case BSG_ERR_EXCEEDS_SCRATCH: return "request exceeds the fixed scratch array of nvfp4_gemm_noalloc";
    default: return "unknown status";
    }
}

}  // extern "C"
