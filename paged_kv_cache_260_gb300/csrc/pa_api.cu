// pa_api.cu -- the C ABI declared in include/pagedattn.h: host-side argument
// checks, per-device state and kernel dispatch.  Nothing here allocates
// device memory or synchronises, except pa_get_device_error().
#include <algorithm>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <mutex>
#include <stdint.h>

#include "pa_cache.h"
#include "pa_internal.h"
#include "pa_prefill_abi.h"
#include "pa_schedule.cuh"
#include "pa_shared.h"
#include "pagedattn.h"

namespace pa {

// Error bits recorded by the kernels (one word per device).
__device__ uint32_t g_device_error;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    int num_sms = 0;
    uint32_t *err = nullptr;   // device address of g_device_error
    size_t smem_optin = 0;     // largest dynamic shared memory per block
    long long l2_bytes = 0;    // L2 cache size
};

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];

struct AttrEntry {
    const void *func;
    int device;
    size_t smem;
};
constexpr int kMaxAttr = 256;
AttrEntry g_attr[kMaxAttr];
int g_attr_count = 0;

struct StaticEntry {
    const void *func;
    int device;
    size_t bytes;              // the kernel's static shared memory
};
constexpr int kMaxStatic = 64;
StaticEntry g_static[kMaxStatic];
int g_static_count = 0;

struct OccEntry {
    const void *func;
    int device;
    size_t smem;
    int blocks;
};
constexpr int kMaxOcc = 512;
OccEntry g_occ[kMaxOcc];
int g_occ_count = 0;

int device_state(DeviceState **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState &st = g_dev[dev];
    if (!st.ready) {
        int sms = 0, optin = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return PA_ERR_CUDA;
        if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
            return PA_ERR_CUDA;
        int l2 = 0;
        if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
            return PA_ERR_CUDA;
        st.l2_bytes = l2;
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_device_error) != cudaSuccess)
            return PA_ERR_CUDA;
        st.num_sms = sms;
        st.smem_optin = (size_t)optin;
        st.err = static_cast<uint32_t *>(addr);
        st.ready = true;
    }
    *out = &st;
    return PA_OK;
}

// Raise the kernel's dynamic shared memory limit once per (device, size).
int ensure_smem(const void *func, int dev, size_t smem)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    for (int i = 0; i < g_attr_count; ++i)
        if (g_attr[i].func == func && g_attr[i].device == dev) {
            if (g_attr[i].smem >= smem)
                return PA_OK;
            if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
                cudaSuccess)
                return PA_ERR_CUDA;
            g_attr[i].smem = smem;
            return PA_OK;
        }
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return PA_ERR_CUDA;
    if (g_attr_count < kMaxAttr)
        g_attr[g_attr_count++] = AttrEntry{func, dev, smem};
    return PA_OK;
}

// Dynamic shared memory a block of this kernel may use on the device: the
// per-block limit less the kernel's static shared memory.
int dynamic_smem_limit(const void *func, int dev, size_t optin, size_t *limit)
{
    size_t bytes = 0;
    bool found = false;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        for (int i = 0; i < g_static_count; ++i)
            if (g_static[i].func == func && g_static[i].device == dev) {
                bytes = g_static[i].bytes;
                found = true;
                break;
            }
    }
    if (!found) {
        cudaFuncAttributes attr{};
        if (cudaFuncGetAttributes(&attr, func) != cudaSuccess)
            return PA_ERR_CUDA;
        bytes = attr.sharedSizeBytes;
        std::lock_guard<std::mutex> lock(g_mutex);
        if (g_static_count < kMaxStatic)
            g_static[g_static_count++] = StaticEntry{func, dev, bytes};
    }
    *limit = bytes < optin ? optin - bytes : 0;
    return PA_OK;
}

int occupancy(const void *func, int dev, int threads, size_t smem, int *blocks)
{
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        for (int i = 0; i < g_occ_count; ++i)
            if (g_occ[i].func == func && g_occ[i].device == dev && g_occ[i].smem == smem) {
                *blocks = g_occ[i].blocks;
                return PA_OK;
            }
    }
    int nb = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, func, threads, smem) != cudaSuccess)
        return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_occ_count < kMaxOcc)
        g_occ[g_occ_count++] = OccEntry{func, dev, smem, nb};
    *blocks = nb;
    return PA_OK;
}

// cuTensorMapEncodeTiled, reached through the runtime so the library needs no
// direct link against the driver library.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// The pool seen as a 2-D array [num_blocks * num_kv_heads * 16 rows][head_dim]
// of 16-bit elements, read in boxes of 16 rows x 64 columns (128 bytes) with
// the 128-byte swizzle.  One box row is one token's 64 channels.
// The pool maps of recent calls: a map is fixed by the pool's address, element
// type, head size and row count, so a serving loop that calls every step on
// the same pools encodes each map once.
struct PoolMapEntry {
    const void *pool;
    int dtype, head_dim;
    long long rows;
    CUtensorMap map;
};
constexpr int kPoolMaps = 8;
PoolMapEntry g_pool_maps[kPoolMaps];
int g_pool_map_count = 0, g_pool_map_next = 0;

int make_pool_map(CUtensorMap *tm, const void *pool, int dtype, int head_dim, long long rows)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    for (int i = 0; i < g_pool_map_count; ++i) {
        const PoolMapEntry &e = g_pool_maps[i];
        if (e.pool == pool && e.dtype == dtype && e.head_dim == head_dim && e.rows == rows) {
            *tm = e.map;
            return PA_OK;
        }
    }
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc)
        return PA_ERR_CUDA;
    const cuuint64_t gdim[2] = {(cuuint64_t)head_dim, (cuuint64_t)rows};
    const cuuint64_t gstride[1] = {(cuuint64_t)head_dim * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kBlockSize};
    const cuuint32_t estride[2] = {1, 1};
    const CUresult r = enc(tm,
                           dtype == PA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                  : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                           2, const_cast<void *>(pool), gdim, gstride, box, estride,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return PA_ERR_CUDA;
    PoolMapEntry &e = g_pool_maps[g_pool_map_next];
    e = PoolMapEntry{pool, dtype, head_dim, rows, *tm};
    g_pool_map_next = (g_pool_map_next + 1) % kPoolMaps;
    if (g_pool_map_count < kPoolMaps)
        ++g_pool_map_count;
    return PA_OK;
}

int launch_dependent(const void *func, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                     void **args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, func, args) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int check_common(int num_kv_heads, int head_dim, int block_size, int num_blocks, int dtype)
{
    if (dtype != PA_DTYPE_F16 && dtype != PA_DTYPE_BF16)
        return PA_ERR_UNSUPPORTED;
    if (block_size != kBlockSize)
        return PA_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128)
        return PA_ERR_UNSUPPORTED;
    if (num_kv_heads <= 0 || num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    return PA_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? PA_OK : PA_ERR_CUDA; }

struct WorkspaceLayout {
    size_t m_off, l_off, o_off, sm_off, sl_off, so_off, desc_off, pre_off, lens_off, share_off,
        blk_off, total;
    bool seq_global;
};

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace of one decode, each array starting at a 256-byte boundary:
//   fixed mode only: m, l, o of every partition, [num_seqs][num_heads][P_max]
//   (x head_dim for o) -- the documented layout;
//   both split modes: m, l, o of two slots per worker and query head of the
//   group (a worker's first and last pieces are the only ones that can be
//   cut), then one cut descriptor per worker;
//   any mode, batches above kSeqsInSmem: the unit prefix [num_seqs + 1] and
//   the clamped lengths [num_seqs], int32, and the first-block-shared flags
//   [num_seqs] plus one "any flag set" byte, built by the prep kernels, and
//   the prep blocks' unit counts and flags [ceil(num_seqs / kPrepSeqs)][2].
WorkspaceLayout workspace_layout(int mode, int num_seqs, int num_heads, int num_kv_heads,
                                 int head_dim, int p_max, int workers)
{
    WorkspaceLayout w{};
    size_t at = 0;
    if (mode != kModeWhole) {
        const int group = num_heads / num_kv_heads;
        const size_t prow = mode == kModeFixed ? (size_t)num_seqs * num_heads * p_max : 0;
        const size_t srow = 2 * (size_t)workers * group;
        w.m_off = at;
        at = round_up(at + sizeof(float) * prow, 256);
        w.l_off = at;
        at = round_up(at + sizeof(float) * prow, 256);
        w.o_off = at;
        at = round_up(at + sizeof(float) * prow * head_dim, 256);
        w.sm_off = at;
        at = round_up(at + sizeof(float) * srow, 256);
        w.sl_off = at;
        at = round_up(at + sizeof(float) * srow, 256);
        w.so_off = at;
        at = round_up(at + sizeof(float) * srow * head_dim, 256);
        w.desc_off = at;
        at = round_up(at + sizeof(CutDesc) * workers, 256);
    }
    if (num_seqs > kSeqsInSmem) {
        w.seq_global = true;
        w.pre_off = at;
        at = round_up(at + sizeof(int32_t) * ((size_t)num_seqs + 1), 256);
        w.lens_off = at;
        at = round_up(at + sizeof(int32_t) * (size_t)num_seqs, 256);
        w.share_off = at;
        at = round_up(at + (size_t)num_seqs + 1, 256);
        w.blk_off = at;
        at = round_up(at + 2 * sizeof(int32_t) * (((size_t)num_seqs + kPrepSeqs - 1) / kPrepSeqs),
                      256);
    }
    w.total = at;
    return w;
}

int decode_mode(int partition_size, int *mode, int *part_tiles)
{
    if (partition_size == -1) {
        *mode = kModeWhole;
        *part_tiles = 1 << 30;
    } else if (partition_size == 0) {
        *mode = kModeBalanced;
        *part_tiles = 0;
    } else if (partition_size > 0 && partition_size % kBlockSize == 0) {
        *mode = kModeFixed;
        *part_tiles = partition_size / kBlockSize;
    } else {
        return PA_ERR_INVALID_ARG;
    }
    return PA_OK;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" {

int pa_version(void) { return PAGEDATTN_VERSION; }

const char *pa_status_string(int status)
{
    switch (status) {
    case PA_OK:
        return "ok";
    case PA_ERR_INVALID_ARG:
        return "invalid argument";
    case PA_ERR_UNSUPPORTED:
        return "unsupported configuration";
    case PA_ERR_WORKSPACE:
        return "workspace missing or too small";
    case PA_ERR_CUDA:
        return "CUDA error";
    case PA_ERR_DEVICE:
        return "a kernel recorded an error";
    default:
        return "unknown status";
    }
}

size_t pa_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                int max_blocks_per_seq, int partition_size)
{
    int mode, pt;
    if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads ||
        max_blocks_per_seq <= 0 || decode_mode(partition_size, &mode, &pt) != PA_OK)
        return 0;
    int workers = 0;
    if (mode != kModeWhole) {
        DeviceState *ds;
        if (device_state(&ds) != PA_OK)
            return 0;
        workers = ds->num_sms * kMaxWarpsPerSM;
    }
    const int p_max = mode == kModeFixed ? (max_blocks_per_seq + pt - 1) / pt : 1;
    return workspace_layout(mode, num_seqs, num_heads, num_kv_heads, head_dim, p_max, workers)
        .total;
}

// Where a balanced decode leaves the pieces of the runs it cut.
struct CutPieces {
    const float *sm = nullptr, *sl = nullptr, *so = nullptr;
};

// What a decode does beyond pa_decode: the fused append, partial outputs.
struct DecodeExtra {
    const void *k_new = nullptr, *v_new = nullptr;
    const int64_t *slot_mapping = nullptr;
    float *out_m = nullptr, *out_l = nullptr, *out_o = nullptr;
    const CUtensorMap *tmk = nullptr, *tmv = nullptr;   // the pools' maps, if already encoded
    // partial outputs, balanced split: record per run whether and where it
    // was cut ([num_seqs][num_kv_heads] pairs of ints) and leave the cut
    // pieces to the caller's merge (no merge_cut); *pieces says where they are
    int32_t *cut_of_run = nullptr;
    CutPieces *pieces = nullptr;
};

static int decode_impl(void *out, const void *q, const void *k_cache, const void *v_cache,
                       const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                       int num_heads, int num_kv_heads, int head_dim, int block_size,
                       int max_blocks_per_seq, int num_blocks, float scale, int dtype,
                       int partition_size, void *workspace, size_t workspace_bytes, void *stream,
                       const DecodeExtra &x)
{
    int rc = check_common(num_kv_heads, head_dim, block_size, num_blocks, dtype);
    if (rc != PA_OK)
        return rc;
    if (num_seqs < 0 || num_heads <= 0 || max_blocks_per_seq <= 0 || !isfinite(scale))
        return PA_ERR_INVALID_ARG;
    if (num_heads % num_kv_heads)
        return PA_ERR_INVALID_ARG;
    const int group = num_heads / num_kv_heads;
    if (group > kMaxGroup)
        return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0)
        return PA_OK;
    if ((!out && !x.out_o) || !q || !k_cache || !v_cache || !block_tables || !seq_lens)
        return PA_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return PA_ERR_INVALID_ARG;
    // flat tile indices and tensor-map row coordinates are 32-bit
    const long long pool_rows = (long long)num_blocks * num_kv_heads * kBlockSize;
    if ((long long)num_seqs * max_blocks_per_seq * num_kv_heads >= (1LL << 31) ||
        (long long)max_blocks_per_seq * kBlockSize >= (1LL << 30) || pool_rows >= (1LL << 31))
        return PA_ERR_UNSUPPORTED;
    int mode, pt;
    rc = decode_mode(partition_size, &mode, &pt);
    if (rc != PA_OK)
        return rc;
    if (x.cut_of_run && (mode == kModeFixed || !x.out_o || !x.pieces))
        return PA_ERR_INVALID_ARG;

    KernelSet ks{};
    bool found;
    if (group <= 8)
        found = dtype == PA_DTYPE_F16 ? decode_kernels_f16(head_dim, &ks)
                                      : decode_kernels_bf16(head_dim, &ks);
    else
        found = dtype == PA_DTYPE_F16 ? decode_kernels_f16_g16(head_dim, &ks)
                                      : decode_kernels_bf16_g16(head_dim, &ks);
    if (!found)
        return PA_ERR_UNSUPPORTED;
    DeviceState *ds;
    rc = device_state(&ds);
    if (rc != PA_OK)
        return rc;
    // Short runs, each on a warp of its own: the balanced split would cut
    // runs of a few tiles and add a merge launch to wait for, while whole
    // runs finish within a few tile loads (a 4 x 100-token batch: 11.7-13.1
    // against 15.4-15.6 us per step)
    if (mode == kModeBalanced && max_blocks_per_seq <= kWholeMaxBlocks &&
        (long long)num_seqs * num_kv_heads <= (long long)kWholeRunsPerSM * ds->num_sms)
        mode = kModeWhole;
    int dev = 0;
    cudaGetDevice(&dev);
    // per-sequence arrays in shared memory up to kSeqsInSmem sequences, else
    // in the workspace (static shared memory counts against the limit too)
    const bool seq_global = num_seqs > kSeqsInSmem;
    size_t limit = 0;
    const size_t smem = seq_global ? ks.smem_fixed : decode_smem_bytes(ks.smem_fixed, num_seqs);
    rc = dynamic_smem_limit(x.out_o && ks.decode_partial ? ks.decode_partial : ks.decode, dev,
                            ds->smem_optin, &limit);
    if (rc != PA_OK)
        return rc;
    if (smem > limit)
        return PA_ERR_UNSUPPORTED;
    const void *decode_fn = x.out_o ? ks.decode_partial : ks.decode;
    if (!decode_fn)
        return PA_ERR_UNSUPPORTED;
    const int warps = ks.warps;
    // Blocks per SM, looked up for the shared memory rounded up to 2 KiB
    // (within the kernel's limit): a serving loop's batch size changes every
    // step, and the rounding keeps the cache of occupancy results to ~100
    // entries per kernel.  A larger footprint can only lower the count, so
    // every block of the grid still fits.  The kernel's dynamic shared
    // memory limit is raised to the rounded figure too, since the occupancy
    // query counts no block that would exceed it.
    const size_t smem_key = std::min(round_up(smem, 2048), limit);
    rc = ensure_smem(decode_fn, dev, smem_key);
    if (rc != PA_OK)
        return rc;
    int per_sm = 0;
    rc = occupancy(decode_fn, dev, warps * 32, smem_key, &per_sm);
    if (rc != PA_OK)
        return rc;
    if (per_sm < 1)
        return PA_ERR_UNSUPPORTED;
    if (per_sm * warps > kMaxWarpsPerSM)
        per_sm = kMaxWarpsPerSM / warps;
    const int grid = ds->num_sms * per_sm;
    const int workers = grid * warps;
    const int p_max = mode == kModeFixed ? (max_blocks_per_seq + pt - 1) / pt : 1;
    // sized for the most workers any call on this device can use, so the
    // size does not depend on the launch configuration chosen here
    const WorkspaceLayout wl = workspace_layout(mode, num_seqs, num_heads, num_kv_heads, head_dim,
                                                p_max, ds->num_sms * kMaxWarpsPerSM);
    if (wl.total > 0 && (!workspace || workspace_bytes < wl.total || !aligned(workspace, 256)))
        return PA_ERR_WORKSPACE;

    DecodeParams p{};
    p.out = out;
    p.q = q;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.k_new = x.k_new;
    p.v_new = x.v_new;
    p.slot_mapping = x.slot_mapping;
    p.out_m = x.out_m;
    p.out_l = x.out_l;
    p.out_o = x.out_o;
    p.cut_of_run = x.cut_of_run;
    char *ws = static_cast<char *>(workspace);
    if (wl.total > 0) {
        p.ws_m = reinterpret_cast<float *>(ws + wl.m_off);
        p.ws_l = reinterpret_cast<float *>(ws + wl.l_off);
        p.ws_o = reinterpret_cast<float *>(ws + wl.o_off);
        p.ws_sm = reinterpret_cast<float *>(ws + wl.sm_off);
        p.ws_sl = reinterpret_cast<float *>(ws + wl.sl_off);
        p.ws_so = reinterpret_cast<float *>(ws + wl.so_off);
        if (mode != kModeWhole)
            p.ws_desc = reinterpret_cast<CutDesc *>(ws + wl.desc_off);
        if (wl.seq_global) {
            p.ws_pre = reinterpret_cast<int32_t *>(ws + wl.pre_off);
            p.ws_lens = reinterpret_cast<int32_t *>(ws + wl.lens_off);
            p.ws_share = reinterpret_cast<uint8_t *>(ws + wl.share_off);
            p.ws_blk = reinterpret_cast<int32_t *>(ws + wl.blk_off);
        }
    }
    p.err = ds->err;
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.max_blocks = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.mode = mode;
    p.part_tiles = pt;
    p.p_max = p_max;
    p.min_tiles = kMinTiles;
    p.workers = workers;
    p.scale_log2 = scale * 1.4426950408889634f;

    CUtensorMap tmk, tmv;
    if (x.tmk && x.tmv) {
        tmk = *x.tmk;
        tmv = *x.tmv;
    } else {
        rc = make_pool_map(&tmk, k_cache, dtype, head_dim, pool_rows);
        if (rc == PA_OK)
            rc = make_pool_map(&tmv, v_cache, dtype, head_dim, pool_rows);
        if (rc != PA_OK)
            return rc;
    }

    // Every kernel here is a programmatic dependent launch: its blocks may be
    // scheduled while the preceding kernel on the stream drains, and they
    // touch no global memory before that kernel has completed.
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void *args[] = {&p, &tmk, &tmv};
    if (wl.seq_global) {
        void *pargs[] = {&p};
        const dim3 pgrid((num_seqs + kPrepSeqs - 1) / kPrepSeqs);
        rc = launch_dependent(ks.prep, pgrid, dim3(kPrepThreads), 0, st, pargs);
        if (rc == PA_OK)
            rc = launch_dependent(ks.prep_fix, pgrid, dim3(kPrepThreads), 0, st, pargs);
        if (rc != PA_OK)
            return rc;
    }
    rc = launch_dependent(decode_fn, dim3(grid), dim3(warps * 32), smem, st, args);
    if (rc != PA_OK || mode == kModeWhole)
        return rc;
    if (x.cut_of_run) {                  // the caller's merge folds the cut pieces
        x.pieces->sm = p.ws_sm;
        x.pieces->sl = p.ws_sl;
        x.pieces->so = p.ws_so;
        return PA_OK;
    }
    void *margs[] = {&p};
    // one warp per query head of the group: small blocks, so all of them can
    // be resident beside the decode while it drains
    rc = launch_dependent(ks.merge_cut, dim3(workers), dim3(32 * group), 0, st, margs);
    if (rc != PA_OK || mode != kModeFixed || p_max < 2)
        return rc;
    return launch_dependent(ks.merge_part, dim3(num_seqs * num_heads), dim3(512), 0, st, margs);
}

int pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
              const int32_t *block_tables, const int32_t *seq_lens, int num_seqs, int num_heads,
              int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
              int num_blocks, float scale, int dtype, int partition_size, void *workspace,
              size_t workspace_bytes, void *stream)
{
    return decode_impl(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs, num_heads,
                       num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, scale,
                       dtype, partition_size, workspace, workspace_bytes, stream, DecodeExtra{});
}

int pa_decode_append(void *out, const void *q, void *k_cache, void *v_cache,
                     const int32_t *block_tables, const int32_t *seq_lens, const void *k_new,
                     const void *v_new, const int64_t *slot_mapping, int num_seqs, int num_heads,
                     int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                     int num_blocks, float scale, int dtype, int partition_size, void *workspace,
                     size_t workspace_bytes, void *stream)
{
    if (num_seqs > 0 && (!k_new || !v_new || !slot_mapping || !aligned(k_new, 16) ||
                         !aligned(v_new, 16) || !aligned(slot_mapping, 8)))
        return PA_ERR_INVALID_ARG;
    DecodeExtra x;
    x.k_new = k_new;
    x.v_new = v_new;
    x.slot_mapping = slot_mapping;
    return decode_impl(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs, num_heads,
                       num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks, scale,
                       dtype, partition_size, workspace, workspace_bytes, stream, x);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// pa_decode_shared_prefix: each group's shared prefix attended by all of the
// group's query columns at once (prefix_attn_kernel, every prefix tile read
// once, in key chunks), the suffixes as one decode over the sequences' own
// tables past the prefix, both with partial outputs, then one log-sum-exp
// merge.
// ---------------------------------------------------------------------------
namespace pa {
namespace {

struct SharedLayout {
    size_t lv, cr, pm, pl, po, xm, xl, xo, dws, dws_bytes, total;
    int cols, col_blocks, chunk_tiles, nchunks;
};

// Key chunks of a prefix of P tiles: enough (group, kv head, column block,
// chunk) thread blocks for about eight per SM (three run at a time), while
// every chunk keeps at least kMinChunkTiles tiles (each chunk adds a partial
// per column to write and merge).
constexpr int kMinChunkTiles = 16;


bool shared_layout(int num_seqs, int group_size, int prefix_len, int num_heads, int num_kv_heads,
                   int head_dim, int max_blocks_per_seq, SharedLayout *L)
{
    if (num_seqs <= 0 || group_size <= 0 || num_seqs % group_size || prefix_len <= 0 ||
        prefix_len % kBlockSize || num_heads <= 0 || num_kv_heads <= 0 ||
        num_heads % num_kv_heads || num_heads / num_kv_heads > kMaxGroup ||
        max_blocks_per_seq <= 0 || prefix_len / kBlockSize > max_blocks_per_seq ||
        (head_dim != 64 && head_dim != 128))
        return false;
    DeviceState *ds;
    if (device_state(&ds) != PA_OK)
        return false;
    const int G = num_heads / num_kv_heads;
    const long long cols = (long long)group_size * G;
    const long long npairs = (long long)(num_seqs / group_size) * num_kv_heads;
    if (cols >= (1LL << 20) || num_seqs >= (1 << 30))
        return false;
    L->cols = (int)cols;
    L->col_blocks = (int)((cols + kPrefixCols - 1) / kPrefixCols);
    const int P = prefix_len / kBlockSize;
    const long long units = npairs * L->col_blocks;
    long long k = (8LL * ds->num_sms + units - 1) / units;
    k = std::max(1LL, std::min(k, (long long)std::max(1, P / kMinChunkTiles)));
    L->chunk_tiles = (int)((P + k - 1) / k);
    L->nchunks = (P + L->chunk_tiles - 1) / L->chunk_tiles;
    if (units * L->nchunks >= (1LL << 31))
        return false;
    const size_t rows = (size_t)num_seqs * num_heads;           // suffix partials
    const size_t xrows = (size_t)L->nchunks * npairs * cols;    // prefix partials
    size_t at = 0;
    auto take = [&](size_t bytes) {
        const size_t off = at;
        at = round_up(at + bytes, 256);
        return off;
    };
    L->lv = take((size_t)num_seqs * sizeof(int32_t));
    L->cr = take((size_t)num_seqs * num_kv_heads * 2 * sizeof(int32_t));
    L->pm = take(rows * sizeof(float));
    L->pl = take(rows * sizeof(float));
    L->po = take(rows * head_dim * sizeof(float));
    L->xm = take(xrows * sizeof(float));
    L->xl = take(xrows * sizeof(float));
    L->xo = take(xrows * head_dim * sizeof(float));
    L->dws_bytes = workspace_layout(kModeBalanced, num_seqs, num_heads, num_kv_heads, head_dim, 1,
                                    ds->num_sms * kMaxWarpsPerSM)
                       .total;
    L->dws = take(L->dws_bytes);
    L->total = at;
    return true;
}

}  // namespace
}  // namespace pa

extern "C" {

size_t pa_decode_shared_prefix_workspace_size(int num_seqs, int group_size, int prefix_len,
                                              int num_heads, int num_kv_heads, int head_dim,
                                              int max_blocks_per_seq)
{
    SharedLayout L;
    if (!shared_layout(num_seqs, group_size, prefix_len, num_heads, num_kv_heads, head_dim,
                       max_blocks_per_seq, &L))
        return 0;
    return L.total;
}

int pa_decode_shared_prefix(void *out, const void *q, void *k_cache, void *v_cache,
                            const int32_t *block_tables, const int32_t *seq_lens,
                            const void *k_new, const void *v_new, const int64_t *slot_mapping,
                            int num_seqs, int group_size, int prefix_len, int num_heads,
                            int num_kv_heads, int head_dim, int block_size,
                            int max_blocks_per_seq, int num_blocks, float scale, int dtype,
                            void *workspace, size_t workspace_bytes, void *stream)
{
    int rc = check_common(num_kv_heads, head_dim, block_size, num_blocks, dtype);
    if (rc != PA_OK)
        return rc;
    if (num_seqs < 0 || num_heads <= 0 || num_heads % num_kv_heads || !isfinite(scale))
        return PA_ERR_INVALID_ARG;
    if (num_heads / num_kv_heads > kMaxGroup)
        return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0)
        return PA_OK;
    const bool append = k_new || v_new || slot_mapping;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens ||
        (append && (!k_new || !v_new || !slot_mapping)))
        return PA_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(block_tables, 4) ||
        !aligned(seq_lens, 4) ||
        (append && (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(slot_mapping, 8))))
        return PA_ERR_INVALID_ARG;
    SharedLayout L;
    if (!shared_layout(num_seqs, group_size, prefix_len, num_heads, num_kv_heads, head_dim,
                       max_blocks_per_seq, &L))
        return PA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < L.total || !aligned(workspace, 256))
        return PA_ERR_WORKSPACE;
    DeviceState *ds;
    rc = device_state(&ds);
    if (rc != PA_OK)
        return rc;
    char *ws = static_cast<char *>(workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    SharedParams sp{};
    sp.num_seqs = num_seqs;
    sp.group_size = group_size;
    sp.prefix_tiles = prefix_len / kBlockSize;
    sp.num_heads = num_heads;
    sp.num_kv_heads = num_kv_heads;
    sp.head_dim = head_dim;
    sp.err = ds->err;
    sp.pm = reinterpret_cast<float *>(ws + L.pm);
    sp.pl = reinterpret_cast<float *>(ws + L.pl);
    sp.po = reinterpret_cast<float *>(ws + L.po);
    sp.xm = reinterpret_cast<float *>(ws + L.xm);
    sp.xl = reinterpret_cast<float *>(ws + L.xl);
    sp.xo = reinterpret_cast<float *>(ws + L.xo);
    sp.nchunks = L.nchunks;
    sp.cols = L.cols;
    sp.out = out;
    // the prefix: every query column of a group over the group's shared
    // blocks, each block read once
    const long long pool_rows = (long long)num_blocks * num_kv_heads * kBlockSize;
    if (pool_rows >= (1LL << 31))
        return PA_ERR_UNSUPPORTED;
    CUtensorMap tmk, tmv;
    rc = make_pool_map(&tmk, k_cache, dtype, head_dim, pool_rows);
    if (rc == PA_OK)
        rc = make_pool_map(&tmv, v_cache, dtype, head_dim, pool_rows);
    if (rc != PA_OK)
        return rc;
    PrefixParams xp{};
    xp.q = q;
    xp.block_tables = block_tables;
    xp.num_heads = num_heads;
    xp.num_kv_heads = num_kv_heads;
    xp.max_blocks = max_blocks_per_seq;
    xp.num_blocks = num_blocks;
    xp.group_size = group_size;
    xp.num_groups = num_seqs / group_size;
    xp.cols = L.cols;
    xp.col_blocks = L.col_blocks;
    xp.prefix_tiles = prefix_len / kBlockSize;
    xp.chunk_tiles = L.chunk_tiles;
    xp.nchunks = L.nchunks;
    xp.scale_log2 = scale * 1.4426950408889634f;
    xp.err = ds->err;
    xp.xm = reinterpret_cast<float *>(ws + L.xm);
    xp.xl = reinterpret_cast<float *>(ws + L.xl);
    xp.xo = reinterpret_cast<float *>(ws + L.xo);
    xp.seq_lens = seq_lens;
    xp.lens_v = reinterpret_cast<int32_t *>(ws + L.lv);
    xp.num_seqs = num_seqs;
    const PrefixKernel pk = prefix_kernel(xp, dtype == PA_DTYPE_BF16, head_dim);
    int dev = 0;
    cudaGetDevice(&dev);
    rc = ensure_smem(pk.fn, dev, pk.smem);
    if (rc != PA_OK)
        return rc;
    void *xargs[] = {&xp, &tmk, &tmv};
    rc = launch_dependent(pk.fn, dim3((unsigned)pk.blocks), dim3(pk.threads), pk.smem, st, xargs);
    if (rc != PA_OK)
        return rc;
    // the suffixes: every sequence's own tokens past the prefix (and its new
    // token), one decode with partial outputs over the sequences' tables from
    // the first block past the prefix on (rows keep their stride)
    DecodeExtra x;
    x.k_new = k_new;
    x.v_new = v_new;
    x.slot_mapping = slot_mapping;
    x.out_m = reinterpret_cast<float *>(ws + L.pm);
    x.out_l = reinterpret_cast<float *>(ws + L.pl);
    x.out_o = reinterpret_cast<float *>(ws + L.po);
    x.tmk = &tmk;
    x.tmv = &tmv;
    // runs the balanced split cuts are folded by the final merge, piece by
    // piece, instead of by a merge of their own
    CutPieces pieces;
    x.cut_of_run = reinterpret_cast<int32_t *>(ws + L.cr);
    x.pieces = &pieces;
    rc = decode_impl(nullptr, q, k_cache, v_cache, block_tables + sp.prefix_tiles, xp.lens_v,
                     num_seqs, num_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                     num_blocks, scale, dtype, 0, ws + L.dws, L.dws_bytes, stream, x);
    if (rc != PA_OK)
        return rc;
    sp.cut_of_run = x.cut_of_run;
    sp.sm = pieces.sm;
    sp.sl = pieces.sl;
    sp.so = pieces.so;
    return cuda_status(launch_shared_merge(sp, dtype == PA_DTYPE_BF16, st));
}

// Query tiles per (sequence, kv head) of a prefill grid, 0 on bad arguments.
static long long prefill_q_ranks(int max_query_len, int num_heads, int num_kv_heads)
{
    if (max_query_len <= 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads ||
        num_heads / num_kv_heads > kPrefillRows)
        return 0;
    const int tokens_per_block = kPrefillTiles * (kPrefillRows / (num_heads / num_kv_heads));
    return (max_query_len + tokens_per_block - 1) / tokens_per_block;
}

// Work-order workspace: the pair count and the order's kind (two ints, 16
// bytes), one word per (sequence, query tile) pair, then each sequence's
// first pair and pair count (int32 each).
size_t pa_prefill_workspace_size(int num_seqs, int max_query_len, int num_heads,
                                 int num_kv_heads)
{
    const long long q_ranks = prefill_q_ranks(max_query_len, num_heads, num_kv_heads);
    if (num_seqs <= 0 || q_ranks <= 0)
        return 0;
    return round_up(16 + 4 * (size_t)num_seqs * (size_t)q_ranks + 8 * (size_t)num_seqs, 256);
}

int pa_prefill(void *out, const void *q, const void *k_cache, const void *v_cache,
               const int32_t *block_tables, const int32_t *seq_lens, const int32_t *query_start,
               int num_seqs, int max_query_len, int num_heads, int num_kv_heads, int head_dim,
               int block_size, int max_blocks_per_seq, int num_blocks, float scale, int dtype,
               void *workspace, size_t workspace_bytes, void *stream)
{
    int rc = check_common(num_kv_heads, head_dim, block_size, num_blocks, dtype);
    if (rc != PA_OK)
        return rc;
    if (num_seqs < 0 || max_query_len < 0 || num_heads <= 0 || max_blocks_per_seq <= 0 ||
        !isfinite(scale) || !(scale > 0.f) || num_heads % num_kv_heads)
        return PA_ERR_INVALID_ARG;
    const int group = num_heads / num_kv_heads;
    if (group > kPrefillRows)
        return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0 || max_query_len == 0)
        return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens || !query_start)
        return PA_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_tables, 4) || !aligned(seq_lens, 4) || !aligned(query_start, 4))
        return PA_ERR_INVALID_ARG;
    const long long pool_rows = (long long)num_blocks * num_kv_heads * kBlockSize;
    const long long q_ranks = prefill_q_ranks(max_query_len, num_heads, num_kv_heads);
    const long long grid = q_ranks * num_seqs * num_kv_heads;
    if ((long long)max_blocks_per_seq * kBlockSize >= (1LL << 30) || pool_rows >= (1LL << 31) ||
        grid >= (1LL << 31))
        return PA_ERR_UNSUPPORTED;
    const bool planned = workspace != nullptr;
    if (planned) {
        // plan entries pack (sequence, tile) into 16 + 16 bits
        if (num_seqs > 65535 || q_ranks > 65535)
            return PA_ERR_UNSUPPORTED;
        if (!aligned(workspace, 256) ||
            workspace_bytes < pa_prefill_workspace_size(num_seqs, max_query_len, num_heads,
                                                        num_kv_heads))
            return PA_ERR_WORKSPACE;
    }
    PrefillKernel kk{};
    if (!prefill_kernel(dtype, head_dim, &kk))
        return PA_ERR_UNSUPPORTED;
    DeviceState *ds;
    rc = device_state(&ds);
    if (rc != PA_OK)
        return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    size_t limit = 0;
    rc = dynamic_smem_limit(kk.fn, dev, ds->smem_optin, &limit);
    if (rc != PA_OK)
        return rc;
    if (kk.smem > limit)
        return PA_ERR_UNSUPPORTED;
    rc = ensure_smem(kk.fn, dev, kk.smem);
    if (rc != PA_OK)
        return rc;
    CUtensorMap tmk, tmv;
    rc = make_pool_map(&tmk, k_cache, dtype, head_dim, pool_rows);
    if (rc == PA_OK)
        rc = make_pool_map(&tmv, v_cache, dtype, head_dim, pool_rows);
    if (rc != PA_OK)
        return rc;
    PrefillParams p{};
    p.out = out;
    p.q = q;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.query_start = query_start;
    p.err = ds->err;
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.max_blocks = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.q_ranks = (int)q_ranks;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.wave = ds->num_sms;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (planned) {
        int *count = static_cast<int *>(workspace);
        int *by_seq = count + 1;
        uint32_t *plan = reinterpret_cast<uint32_t *>(static_cast<char *>(workspace) + 16);
        int32_t *seq_start = reinterpret_cast<int32_t *>(plan + (size_t)num_seqs * q_ranks);
        int32_t *seq_nq = seq_start + num_seqs;
        p.plan = plan;
        p.plan_count = count;
        p.plan_by_seq = by_seq;
        p.plan_seq_start = seq_start;
        p.plan_seq_nq = seq_nq;
        int tpb = kPrefillTiles * (kPrefillRows / group), bn = kPrefillKeys;
        // K and V bytes a token holds over all kv heads, and the L2 size: the
        // plan keeps each sequence's tiles together when the batch's K/V
        // does not fit in L2
        long long kv_bytes_per_token = 2LL * num_kv_heads * head_dim * 2, l2_bytes = ds->l2_bytes;
        void *pargs[] = {&p,        &tpb,     &bn,       &plan,  &count, &kv_bytes_per_token,
                         &l2_bytes, &by_seq, &seq_start, &seq_nq};
        rc = cuda_status(cudaLaunchKernel(kk.plan_fn, dim3(1), dim3(1024), pargs, 0, st));
        if (rc != PA_OK)
            return rc;
    }
    // a programmatic dependent launch: its blocks may be scheduled while the
    // plan finishes and read no global memory before it has completed
    void *args[] = {&p, &tmk, &tmv};
    return launch_dependent(kk.fn, dim3((unsigned)grid), dim3(kk.threads), kk.smem, st, args);
}

int pa_reshape_and_cache(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                         const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int num_blocks, int dtype, void *stream)
{
    int rc = check_common(num_kv_heads, head_dim, block_size, num_blocks, dtype);
    if (rc != PA_OK)
        return rc;
    if (num_tokens < 0)
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0)
        return PA_OK;
    if (!k_new || !v_new || !k_cache || !v_cache || !slot_mapping)
        return PA_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16) || !aligned(slot_mapping, 8))
        return PA_ERR_INVALID_ARG;
    DeviceState *ds;
    rc = device_state(&ds);
    if (rc != PA_OK)
        return rc;
    return cuda_status(launch_reshape_and_cache(k_new, v_new, k_cache, v_cache, slot_mapping,
                                                num_tokens, num_kv_heads, head_dim, num_blocks,
                                                ds->err, ds->num_sms,
                                                static_cast<cudaStream_t>(stream)));
}

int pa_copy_blocks(void *k_cache, void *v_cache, const int64_t *block_mapping, int num_pairs,
                   int num_kv_heads, int head_dim, int block_size, int num_blocks, int dtype,
                   void *stream)
{
    int rc = check_common(num_kv_heads, head_dim, block_size, num_blocks, dtype);
    if (rc != PA_OK)
        return rc;
    if (num_pairs < 0)
        return PA_ERR_INVALID_ARG;
    if (num_pairs == 0)
        return PA_OK;
    if (!k_cache || !v_cache || !block_mapping)
        return PA_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(block_mapping, 8))
        return PA_ERR_INVALID_ARG;
    DeviceState *ds;
    rc = device_state(&ds);
    if (rc != PA_OK)
        return rc;
    return cuda_status(launch_copy_blocks(k_cache, v_cache, k_cache, v_cache, block_mapping,
                                          num_pairs, num_kv_heads, head_dim, num_blocks,
                                          num_blocks, ds->err, static_cast<cudaStream_t>(stream)));
}

// Device address of a pool the kernels may read or write: device or managed
// memory, or host memory that is page-locked and mapped; nullptr otherwise.
static void *device_view(void *p)
{
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();   // keep the failed query out of later error checks
        return nullptr;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged ||
        a.type == cudaMemoryTypeHost)
        return a.devicePointer;
    return nullptr;
}

int pa_swap_blocks(void *dst_k, void *dst_v, const void *src_k, const void *src_v,
                   const int64_t *block_mapping, int num_pairs, int num_kv_heads, int head_dim,
                   int block_size, int src_num_blocks, int dst_num_blocks, int dtype, void *stream)
{
    int rc = check_common(num_kv_heads, head_dim, block_size, src_num_blocks, dtype);
    if (rc != PA_OK)
        return rc;
    if (num_pairs < 0 || dst_num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_pairs == 0)
        return PA_OK;
    if (!dst_k || !dst_v || !src_k || !src_v || !block_mapping)
        return PA_ERR_INVALID_ARG;
    if (!aligned(dst_k, 16) || !aligned(dst_v, 16) || !aligned(src_k, 16) ||
        !aligned(src_v, 16) || !aligned(block_mapping, 8))
        return PA_ERR_INVALID_ARG;
    DeviceState *ds;
    rc = device_state(&ds);
    if (rc != PA_OK)
        return rc;
    void *dk = device_view(dst_k), *dv = device_view(dst_v);
    void *sk = device_view(const_cast<void *>(src_k)), *sv = device_view(const_cast<void *>(src_v));
    void *bm = device_view(const_cast<int64_t *>(block_mapping));
    if (!dk || !dv || !sk || !sv || !bm)
        return PA_ERR_INVALID_ARG;     // pageable host memory: not reachable by the kernel
    return cuda_status(launch_copy_blocks(dk, dv, sk, sv, static_cast<const int64_t *>(bm),
                                          num_pairs, num_kv_heads, head_dim, src_num_blocks,
                                          dst_num_blocks, ds->err,
                                          static_cast<cudaStream_t>(stream)));
}

int pa_gather_kv(void *k_out, void *v_out, const void *k_cache, const void *v_cache,
                 const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                 int num_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                 int num_blocks, int dtype, void *stream)
{
    int rc = check_common(num_kv_heads, head_dim, block_size, num_blocks, dtype);
    if (rc != PA_OK)
        return rc;
    if (num_seqs < 0 || max_blocks_per_seq <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0)
        return PA_OK;
    if (!k_out || !v_out || !k_cache || !v_cache || !block_tables || !seq_lens)
        return PA_ERR_INVALID_ARG;
    if (!aligned(k_out, 16) || !aligned(v_out, 16) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16) || !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return PA_ERR_INVALID_ARG;
    DeviceState *ds;
    rc = device_state(&ds);
    if (rc != PA_OK)
        return rc;
    return cuda_status(launch_gather_kv(k_out, v_out, k_cache, v_cache, block_tables, seq_lens,
                                        num_seqs, num_kv_heads, head_dim, max_blocks_per_seq,
                                        num_blocks, ds->err, ds->num_sms,
                                        static_cast<cudaStream_t>(stream)));
}

int pa_validate_tables(const int32_t *block_tables, const int32_t *seq_lens, int num_seqs,
                       int max_blocks_per_seq, int num_blocks, int block_size,
                       uint32_t *bad_count, void *stream)
{
    if (block_size != kBlockSize)
        return PA_ERR_UNSUPPORTED;
    if (num_seqs < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0)
        return PA_OK;
    if (!block_tables || !seq_lens || !bad_count || !aligned(block_tables, 4) ||
        !aligned(seq_lens, 4) || !aligned(bad_count, 4))
        return PA_ERR_INVALID_ARG;
    DeviceState *ds;
    int rc = device_state(&ds);
    if (rc != PA_OK)
        return rc;
    return cuda_status(launch_validate_tables(block_tables, seq_lens, num_seqs, max_blocks_per_seq,
                                              num_blocks, bad_count, ds->num_sms,
                                              static_cast<cudaStream_t>(stream)));
}

int pa_selftest_bounded_wait(int limit_us, void *stream)
{
    if (limit_us <= 0 || limit_us > 1000000)
        return PA_ERR_INVALID_ARG;
    DeviceState *ds;
    int rc = device_state(&ds);
    if (rc != PA_OK)
        return rc;
    return cuda_status(launch_bounded_wait_selftest((uint64_t)limit_us * 1000, ds->err,
                                                    static_cast<cudaStream_t>(stream)));
}

int pa_get_device_error(void *stream, uint32_t *bits, int clear)
{
    if (!bits)
        return PA_ERR_INVALID_ARG;
    DeviceState *ds;
    int rc = device_state(&ds);
    if (rc != PA_OK)
        return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t host = 0;
    if (cudaMemcpyAsync(&host, ds->err, sizeof host, cudaMemcpyDeviceToHost, st) != cudaSuccess)
        return PA_ERR_CUDA;
    if (clear && cudaMemsetAsync(ds->err, 0, sizeof(uint32_t), st) != cudaSuccess)
        return PA_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess)
        return PA_ERR_CUDA;
    *bits = host;
    return host ? PA_ERR_DEVICE : PA_OK;
}

}  // extern "C"
