// extern "C" entry points of libpagedkv.so: argument validation, tensor-map
// encoding, partition sizing and kernel dispatch.  Declarations and the contract
// of every function are in include/pagedkv.h.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <random>
#include <tuple>
#include <vector>

#include "pa_internal.h"

#include <initializer_list>

#ifndef PA_L2_PROMOTION
#define PA_L2_PROMOTION CU_TENSOR_MAP_L2_PROMOTION_L2_256B
#endif

namespace pagedkv {

namespace {

__device__ unsigned int g_device_errors;  // PA_DEVERR_* flags raised by kernels

thread_local int t_last_cuda_error = 0;

pa_status cuda_fail(cudaError_t e)
{
    t_last_cuda_error = (int)e;
    cudaGetLastError();  // clear the sticky launch error of this thread
    return PA_ERR_CUDA;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int elem_size(pa_dtype d) { return d == PA_F32 ? 4 : 2; }

bool dtype_ok(int d) { return d == PA_F32 || d == PA_F16 || d == PA_BF16; }

std::mutex g_mu;

// ---- per-device facts ----------------------------------------------------------
std::map<int, int> g_sm_count;
std::map<std::tuple<void *, int, size_t>, int> g_occupancy;
std::map<std::pair<void *, int>, size_t> g_smem_limit;
std::map<int, unsigned int *> g_err_ptr;

unsigned int *device_error_word(int dev, cudaError_t *err)
{
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_err_ptr.find(dev);
    if (it != g_err_ptr.end())
        return it->second;
    void *ptr = nullptr;
    *err = cudaGetSymbolAddress(&ptr, g_device_errors);
    if (*err != cudaSuccess)
        return nullptr;
    g_err_ptr[dev] = static_cast<unsigned int *>(ptr);
    return static_cast<unsigned int *>(ptr);
}

// ---- tensor maps ---------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        cudaGetLastError();
    });
    return fn;
}

// Cache [num_blocks][B][Hkv][d] seen as 4-D: (element within a 128-byte row of d,
// token slot, 128-byte row of d, kv head).  One box = one kv head of one block:
// its B token rows, each d / (128 bytes) rows of 128 bytes, landing chunk-major
// (all tokens' first 128 bytes of d, then the next), with 128-byte swizzle.
// With `vbase` (above `base`, a multiple of 16 bytes away) a fifth dimension of
// extent 2 steps from the K cache to the V cache: one box is then a block's K tile
// followed by its V tile.
bool make_cache_map(CUtensorMap *map, const void *base, const void *vbase, pa_dtype dt,
                    int num_blocks, int B, int Hkv, int D)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    const int es = elem_size(dt);
    const int ce = 128 / es;
    const uintptr_t kv_gap = vbase ? (uintptr_t)vbase - (uintptr_t)base : 0;
    const cuuint32_t rank = vbase ? 5 : 4;
    const cuuint64_t dims[5] = {(cuuint64_t)ce, (cuuint64_t)num_blocks * (cuuint64_t)B,
                                (cuuint64_t)(D / ce), (cuuint64_t)Hkv, 2};
    const cuuint64_t strides[4] = {(cuuint64_t)Hkv * D * es, 128, (cuuint64_t)D * es,
                                   (cuuint64_t)kv_gap};
    const cuuint32_t box[5] = {(cuuint32_t)ce, (cuuint32_t)B, (cuuint32_t)(D / ce), 1, 2};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUtensorMapDataType tdt = dt == PA_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                    : dt == PA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const CUresult r = enc(map, tdt, rank, const_cast<void *>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           (CUtensorMapL2promotion)PA_L2_PROMOTION, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Whether one tensor map can step from the K cache to the V cache: V above K, a
// multiple of 16 bytes away, within the 2^40-byte stride limit.  (Caches allocated
// as one [2][num_blocks][B][Hkv][d] buffer always qualify.)
bool kv_joint_ok(const void *k, const void *v)
{
    const uintptr_t a = (uintptr_t)k, b = (uintptr_t)v;
    return b > a && (b - a) % 16 == 0 && (b - a) < (1ull << 40);
}

// ---- partition sizing ------------------------------------------------------------
bool decode_shape_ok(int num_seqs, int Hq, int Hkv, int D, int B, int max_blocks, int part)
{
    if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_blocks <= 0)
        return false;
    if (D != 64 && D != 128)
        return false;
    if (B != 16 && B != 32)
        return false;
    if (part < 0 || (part > 0 && part % B != 0))
        return false;
    if ((long long)max_blocks * B >= (1ll << 31))
        return false;
    return true;
}

// Fixed partitions: a partition size at least as long as the table means one
// partition per sequence.
int resolve_partition(int B, int max_blocks, int part)
{
    const long long max_ctx = (long long)max_blocks * B;
    return part >= max_ctx ? (int)(((max_ctx + B - 1) / B) * B) : part;
}

// Balanced split workspace: one merge counter per CTA, then partial rows for
// 2 slots x 16 query heads per CTA.
size_t balanced_ctas(int sms) { return (size_t)kMaxCtasPerSm * (size_t)sms; }
size_t balanced_rows(int sms) { return 2 * balanced_ctas(sms) * kHeadsPerItem; }
size_t counter_bytes(int sms) { return (balanced_ctas(sms) * 8 + 255) & ~size_t(255); }

// Tags of the merge counters: a process starts from a random value, so that a
// value a workspace kept from another process is unlikely to match.
std::atomic<unsigned int> g_epoch{std::random_device{}()};

// Limit of the device-side waits of decode launches (pa_set_wait_limit_ns).
std::atomic<unsigned long long> g_wait_limit_ns{kWaitTimeoutNs};

unsigned int next_epoch()
{
    unsigned int e = ++g_epoch;
    if (e == 0)  // a zeroed counter must never match
        e = ++g_epoch;
    return e;
}

int current_sms()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return sm_count(dev);
}

}  // namespace

void note_cuda_error(cudaError_t e) { cuda_fail(e); }

unsigned long long wait_limit_ns() { return g_wait_limit_ns.load(); }

int sm_count(int device)
{
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_sm_count.find(device);
    if (it != g_sm_count.end())
        return it->second;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    g_sm_count[device] = n;
    return n;
}

int cached_occupancy(void *kernel, int device, size_t smem, size_t max_smem)
{
    std::lock_guard<std::mutex> lk(g_mu);
    const auto key = std::make_tuple(kernel, device, smem);
    auto it = g_occupancy.find(key);
    if (it != g_occupancy.end())
        return it->second;
    // configurations past the device's per-block opt-in limit cannot launch; the
    // attribute is raised to the largest configuration that can
    int optin = 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) !=
        cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (smem > (size_t)optin)
        return 0;
    if (max_smem > (size_t)optin)
        max_smem = (size_t)optin;
    const auto lkey = std::make_pair(kernel, device);
    if (g_smem_limit[lkey] < max_smem) {
        if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)max_smem) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        g_smem_limit[lkey] = max_smem;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, smem) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    g_occupancy[key] = n;
    return n;
}

}  // namespace pagedkv

using namespace pagedkv;

extern "C" {

const char *pa_status_string(pa_status s)
{
    switch (s) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_OOM: return "out of blocks";
    case PA_ERR_TIMEOUT: return "device wait timed out";
    }
    return "unknown status";
}

int pa_last_cuda_error(void) { return t_last_cuda_error; }

int pa_decode_partition_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                             int block_size, int max_blocks_per_seq, int partition_size)
{
    if (!decode_shape_ok(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                         max_blocks_per_seq, partition_size))
        return -1;
    return partition_size == 0 ? 0 : resolve_partition(block_size, max_blocks_per_seq, partition_size);
}

size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                int block_size, int max_blocks_per_seq, int partition_size)
{
    const int part = pa_decode_partition_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                              block_size, max_blocks_per_seq, partition_size);
    if (part < 0)
        return (size_t)-1;
    if (part == 0) {
        int sms = current_sms();
        sms = sms > 0 ? sms : 160;
        const size_t rows = balanced_rows(sms);
        return counter_bytes(sms) + ((rows * (size_t)head_dim * 4 + 255) & ~size_t(255)) + rows * 4;
    }
    const long long pb = part / block_size;
    const long long parts = (max_blocks_per_seq + pb - 1) / pb;
    if (parts <= 1)
        return 0;
    const size_t rows = (size_t)num_seqs * (size_t)parts * (size_t)num_q_heads;
    size_t bytes = rows * (size_t)head_dim * 4;
    bytes = (bytes + 255) & ~size_t(255);
    return bytes + rows * 4;
}

}  // extern "C"

namespace {

size_t prefix_buffer_bytes(int num_seqs, int num_q_heads, int head_dim)
{
    const size_t rows = (size_t)num_seqs * num_q_heads;
    return (rows * (size_t)(head_dim + 4) * 4 + 255) & ~size_t(255);
}

// pa_decode, pa_decode_append and pa_decode_shared: k_new/v_new null for a plain
// decode; share null unless the batch declares shared-prefix groups.
pa_status decode_impl(void *out, const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *context_lens, int num_seqs, int num_blocks, float scale,
                      int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                      pa_dtype dtype, int partition_size, void *workspace, size_t workspace_bytes,
                      const void *k_new, const void *v_new, void *stream,
                      const int32_t *share = nullptr, const int32_t *plan = nullptr,
                      int plan_grid = 0)
{
    if (num_seqs == 0)
        return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens)
        return PA_ERR_INVALID;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return PA_ERR_INVALID;
    if (num_seqs < 0 || num_blocks <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
        max_blocks_per_seq <= 0 || num_q_heads % num_kv_heads != 0)
        return PA_ERR_INVALID;
    if (partition_size < 0 || (partition_size > 0 && partition_size % block_size != 0))
        return PA_ERR_INVALID;
    if (!dtype_ok(dtype))
        return PA_ERR_UNSUPPORTED;
    if ((head_dim != 64 && head_dim != 128) || (block_size != 16 && block_size != 32))
        return PA_ERR_UNSUPPORTED;
    if ((long long)num_blocks * block_size >= (1ll << 31) ||
        (long long)max_blocks_per_seq * block_size >= (1ll << 31))
        return PA_ERR_INVALID;

    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess)
        return cuda_fail(ce);
    const int sms = sm_count(dev);
    if (sms <= 0)
        return cuda_fail(cudaErrorNoDevice);

    const bool balanced = partition_size == 0;
    const int part = balanced ? 0 : resolve_partition(block_size, max_blocks_per_seq, partition_size);
    const int pb = balanced ? max_blocks_per_seq : part / block_size;
    const int parts = balanced ? 1 : (max_blocks_per_seq + pb - 1) / pb;
    size_t need = pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                           max_blocks_per_seq, partition_size);
    if (need == (size_t)-1)
        return PA_ERR_INVALID;
    const bool shared = share != nullptr && balanced && num_q_heads / num_kv_heads <= kHeadsPerItem;
    // the shared-prefix passes may run at the same time (pass 0 overlaps the end of
    // pass 1), so each has its own merge counters and partial slots
    const size_t pass1_at = need;
    if (shared)
        need += need;
    const size_t pfx_at = need;
    if (shared)
        need += prefix_buffer_bytes(num_seqs, num_q_heads, head_dim);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 16)))
        return PA_ERR_INVALID;
    char *const ws_base = static_cast<char *>(workspace);
    float *pfx = shared ? reinterpret_cast<float *>(ws_base + pfx_at) : nullptr;

    DecodeLaunch L;
    std::memset(&L, 0, sizeof L);
    DecodeParams &p = L.p;
    p.out = out;
    p.q = q;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    if (balanced || parts > 1) {
        const size_t rows =
            balanced ? balanced_rows(sms) : (size_t)num_seqs * parts * num_q_heads;
        if (balanced) {
            p.counters = static_cast<unsigned long long *>(workspace);
            p.epoch = next_epoch();
            workspace = static_cast<char *>(workspace) + counter_bytes(sms);
        }
        p.part_o = static_cast<float *>(workspace);
        p.part_lse = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                               ((rows * head_dim * 4 + 255) & ~size_t(255)));
    }
    p.errors = device_error_word(dev, &ce);
    if (!p.errors)
        return cuda_fail(ce);
    p.wait_ns = wait_limit_ns();
    // a plan holds one entry per CTA of the grid it was made for (the shared-prefix
    // decode's: pass 1's entries, then pass 0's); the launch must use that grid
    p.plan = (balanced && share == nullptr) ? plan : nullptr;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.num_seqs = num_seqs;
    p.max_blocks = max_blocks_per_seq;
    p.num_blocks = num_blocks;
    p.num_q_heads = num_q_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = num_q_heads / num_kv_heads;
    p.head_groups = (p.group + kHeadsPerItem - 1) / kHeadsPerItem;
    p.partition_blocks = pb;
    p.max_parts = parts;
    p.balanced = balanced ? 1 : 0;
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_cache = const_cast<void *>(k_cache);
    p.v_cache = const_cast<void *>(v_cache);
    L.head_dim = head_dim;
    L.block_size = block_size;
    L.sm_count = sms;
    L.grid = plan ? plan_grid : 0;  // 0: the occupancy-sized persistent grid
    // one copy per block for K and V where the caches' placement allows it (the
    // joint map), else one per cache
    p.kv_joint = kv_joint_ok(k_cache, v_cache) &&
                         make_cache_map(&L.tmap_k, k_cache, v_cache, dtype, num_blocks, block_size,
                                        num_kv_heads, head_dim)
                     ? 1
                     : 0;
    if ((!p.kv_joint && !make_cache_map(&L.tmap_k, k_cache, nullptr, dtype, num_blocks, block_size,
                                        num_kv_heads, head_dim)) ||
        !make_cache_map(&L.tmap_v, v_cache, nullptr, dtype, num_blocks, block_size, num_kv_heads,
                        head_dim))
        return cuda_fail(cudaErrorInvalidValue);

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    auto launch = [&](const DecodeLaunch &l) {
        return dtype == PA_F32   ? launch_decode_f32(l, st)
               : dtype == PA_F16 ? launch_decode_f16(l, st)
                                 : launch_decode_bf16(l, st);
    };
    if (shared) {
        // pass 1: every group's shared blocks once, all members' rows at a time
        DecodeLaunch L1 = L;
        char *w1 = ws_base + pass1_at;
        L1.p.counters = reinterpret_cast<unsigned long long *>(w1);
        L1.p.part_o = reinterpret_cast<float *>(w1 + counter_bytes(sms));
        L1.p.part_lse = reinterpret_cast<float *>(
            w1 + counter_bytes(sms) +
            ((balanced_rows(sms) * (size_t)head_dim * 4 + 255) & ~size_t(255)));
        L1.p.pass = 1;
        L1.p.share = share;
        L1.p.pfx = pfx;
        L1.p.k_new = nullptr;
        L1.p.v_new = nullptr;
        L1.p.plan = plan;
        cudaError_t e = launch(L1);
        if (e != cudaSuccess)
            return cuda_fail(e);
        // pass 0: each sequence's own blocks (and newest token), merged with pass 1
        L.p.pass = 0;
        L.p.share = share;
        L.p.pfx = pfx;
        L.p.epoch = next_epoch();
        L.p.plan = plan ? plan + (size_t)plan_grid * kPlanInts : nullptr;
    }
    cudaError_t e = launch(L);
    if (e != cudaSuccess)
        return cuda_fail(e);
    return PA_OK;
}

}  // namespace

extern "C" {

pa_status pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *block_tables, int max_blocks_per_seq,
                    const int32_t *context_lens, int num_seqs, int num_blocks, float scale,
                    int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                    pa_dtype dtype, int partition_size, void *workspace, size_t workspace_bytes,
                    void *stream)
{
    return decode_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                       num_seqs, num_blocks, scale, num_q_heads, num_kv_heads, head_dim, block_size,
                       dtype, partition_size, workspace, workspace_bytes, nullptr, nullptr, stream);
}

pa_status pa_decode_append(void *out, const void *q, void *k_cache, void *v_cache,
                           const void *k_new, const void *v_new, const int32_t *block_tables,
                           int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                           int num_blocks, float scale, int num_q_heads, int num_kv_heads,
                           int head_dim, int block_size, pa_dtype dtype, int partition_size,
                           void *workspace, size_t workspace_bytes, void *stream)
{
    if (num_seqs != 0 && (!k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16)))
        return PA_ERR_INVALID;
    return decode_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                       num_seqs, num_blocks, scale, num_q_heads, num_kv_heads, head_dim, block_size,
                       dtype, partition_size, workspace, workspace_bytes, k_new, v_new, stream);
}

}  // extern "C"

namespace {

// Persistent grid of the planned decode's kernel instance on the current device
// (0: cannot launch or no device).
int plan_grid_for(pa_dtype dtype, int num_q_heads, int num_kv_heads, int head_dim, int block_size)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    const int sms = sm_count(dev);
    if (sms <= 0)
        return 0;
    static const int32_t kSelectPlanned = 0;  // any non-null plan selects the instance
    DecodeLaunch L;
    std::memset(&L, 0, sizeof L);
    L.p.plan = &kSelectPlanned;
    L.p.balanced = 1;
    L.p.num_q_heads = num_q_heads;
    L.p.num_kv_heads = num_kv_heads;
    L.p.group = num_q_heads / num_kv_heads;
    L.p.head_groups = (L.p.group + kHeadsPerItem - 1) / kHeadsPerItem;
    L.head_dim = head_dim;
    L.block_size = block_size;
    L.sm_count = sms;
    L.grid = 0;
    return dtype == PA_F32 ? plan_grid_f32(L) : dtype == PA_F16 ? plan_grid_f16(L) : plan_grid_bf16(L);
}

bool plan_args_ok(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                  int max_blocks_per_seq, int dtype)
{
    return dtype_ok(dtype) && num_seqs >= 0 &&
           decode_shape_ok(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                           max_blocks_per_seq, 0);
}

}  // namespace

extern "C" {

size_t pa_decode_plan_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, int max_blocks_per_seq, pa_dtype dtype)
{
    if (!plan_args_ok(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                      dtype))
        return (size_t)-1;
    const int grid = plan_grid_for(dtype, num_q_heads, num_kv_heads, head_dim, block_size);
    if (grid <= 0)
        return (size_t)-1;
    return (size_t)grid * kPlanInts * sizeof(int32_t);
}

pa_status pa_decode_plan(int32_t *plan, size_t plan_bytes, const int32_t *block_tables,
                         int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                         int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                         pa_dtype dtype)
{
    if (!plan || (num_seqs > 0 && (!block_tables || !context_lens)))
        return PA_ERR_INVALID;
    if (!plan_args_ok(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                      dtype))
        return PA_ERR_INVALID;
    // one entry per CTA of the persistent grid: the plan's size gives the grid
    const size_t entry = (size_t)kPlanInts * sizeof(int32_t);
    if (plan_bytes == 0 || plan_bytes % entry != 0 || plan_bytes / entry > (1u << 20))
        return PA_ERR_INVALID;
    const int grid = (int)(plan_bytes / entry);
    // the stream of the plain balanced split, as the kernel's walk builds it:
    // sequence s contributes U units of kUnitCost + ceil(nb_s / bps) positions
    const int W = max_blocks_per_seq, B = block_size;
    const long long U = (long long)num_kv_heads * ((num_q_heads / num_kv_heads + kHeadsPerItem - 1) /
                                                   kHeadsPerItem);
    const int bps = blocks_per_stage(dtype == PA_F32 ? 4 : 2, B);
    std::vector<long long> start((size_t)num_seqs + 1, 0);
    std::vector<int> len((size_t)num_seqs), ns((size_t)num_seqs);
    for (int s = 0; s < num_seqs; ++s) {
        const long long t = context_lens[s];
        len[s] = (int)std::min<long long>(std::max<long long>(t, 0), (long long)W * B);
        const int nb = (len[s] + B - 1) / B;
        ns[s] = (nb + bps - 1) / bps;
        start[s + 1] = start[s] + U * (kUnitCost + ns[s]);
    }
    const long long total = start[num_seqs];
    const int div = balanced_divisor(total, (long long)num_seqs * U);
    const long long G = num_seqs > 0 ? balanced_grid_of(total, div, grid) : 0;
    std::memset(plan, 0, (size_t)grid * kPlanInts * sizeof(int32_t));
    auto put64 = [](int32_t *e, int f, long long v) {
        e[f] = (int32_t)(uint32_t)(v & 0xffffffffll);
        e[f + 1] = (int32_t)(v >> 32);
    };
    for (int c = 0; c < grid; ++c) {
        int32_t *e = plan + (size_t)c * kPlanInts;
        e[kPlanSeq] = -1;
        put64(e, kPlanTotal, total);
        e[kPlanDiv] = div;
        e[kPlanG] = (int32_t)G;
        e[kPlanGrid] = grid;
        e[kPlanSeqs] = num_seqs;
        if (c >= G)
            continue;
        const long long s_c = c * total / G, e_c = (c + 1) * total / G;
        // the sequence whose positions hold s_c
        const int s = (int)(std::upper_bound(start.begin(), start.end(), s_c) - start.begin()) - 1;
        const long long base = start[s];
        e[kPlanSeq] = s;
        put64(e, kPlanBase, base);
        e[kPlanLen] = len[s];
        put64(e, kPlanStart, s_c);
        put64(e, kPlanEnd, e_c);
        // the first item's first block, when it is in unit (s_c - base) / span of s
        const long long span = kUnitCost + ns[s];
        const long long a = base + (s_c > base ? (s_c - base) / span : 0) * span;
        const long long ra = a + kUnitCost;
        const int nb = (len[s] + B - 1) / B;
        const int j0 = (int)std::min<long long>((std::max(ra, s_c) - ra) * bps, nb);
        e[kPlanJ0] = j0;
        for (int k = 0; k < kPlanWindow; ++k) {
            const int j = j0 + k;
            e[kPlanBlocks + k] = j < W ? block_tables[(size_t)s * W + j] : -1;
        }
    }
    return PA_OK;
}

pa_status pa_decode_planned(void *out, const void *q, void *k_cache, void *v_cache,
                            const void *k_new, const void *v_new, const int32_t *block_tables,
                            int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                            int num_blocks, float scale, int num_q_heads, int num_kv_heads,
                            int head_dim, int block_size, pa_dtype dtype, const int32_t *plan,
                            size_t plan_bytes, void *workspace, size_t workspace_bytes, void *stream)
{
    if (num_seqs == 0)
        return PA_OK;
    if ((k_new == nullptr) != (v_new == nullptr) ||
        (k_new && (!aligned(k_new, 16) || !aligned(v_new, 16))))
        return PA_ERR_INVALID;
    if (!plan || !aligned(plan, 16))
        return PA_ERR_INVALID;
    const size_t need = pa_decode_plan_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                             block_size, max_blocks_per_seq, dtype);
    if (need == (size_t)-1) {
        // invalid sizes: let the common validation report them
        return decode_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                           context_lens, num_seqs, num_blocks, scale, num_q_heads, num_kv_heads,
                           head_dim, block_size, dtype, 0, workspace, workspace_bytes, k_new, v_new,
                           stream);
    }
    if (plan_bytes != need)
        return PA_ERR_INVALID;
    return decode_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                       num_seqs, num_blocks, scale, num_q_heads, num_kv_heads, head_dim, block_size,
                       dtype, 0, workspace, workspace_bytes, k_new, v_new, stream, nullptr, plan,
                       (int)(plan_bytes / (kPlanInts * sizeof(int32_t))));
}

}  // extern "C"

namespace {

// One pass of the balanced split as the kernel's walk builds it: sequence s has
// n[s] units of kUnitCost + ns[s] positions over blocks [first[s], nb[s]) of the
// table row of sequence s; len[s] and aux[s] go to its plan entry.
struct PassStream {
    std::vector<int> n, ns, first, nb, len, aux;
    bool unit_major = false;  // (unit, sequence) order: every n[s] is the same
};

// The plan entries of one pass for a grid of `grid` CTAs (see pa_decode_plan).
void fill_pass_plan(int32_t *plan, int grid, const PassStream &ps, const int32_t *block_tables,
                    int W, int bps)
{
    const int S = (int)ps.n.size();
    auto put64 = [](int32_t *e, int f, long long v) {
        e[f] = (int32_t)(uint32_t)(v & 0xffffffffll);
        e[f + 1] = (int32_t)(v >> 32);
    };
    std::vector<long long> span((size_t)S), start((size_t)S + 1, 0), cum((size_t)S + 1, 0);
    long long units = 0;
    for (int s = 0; s < S; ++s) {
        span[s] = kUnitCost + ps.ns[s];
        start[s + 1] = start[s] + (long long)ps.n[s] * span[s];
        cum[s + 1] = cum[s] + span[s];  // one unit of every sequence (unit-major rows)
        units += ps.n[s];
    }
    const long long total = start[S];
    const int div = balanced_divisor(total, units);
    const long long G = S > 0 ? balanced_grid_of(total, div, grid) : 0;
    const long long U = S > 0 ? ps.n[0] : 0;
    const long long Wrow = ps.unit_major && U > 0 ? total / U : 0;
    std::memset(plan, 0, (size_t)grid * kPlanInts * sizeof(int32_t));
    for (int c = 0; c < grid; ++c) {
        int32_t *e = plan + (size_t)c * kPlanInts;
        e[kPlanSeq] = -1;
        put64(e, kPlanTotal, total);
        e[kPlanDiv] = div;
        e[kPlanG] = (int32_t)G;
        e[kPlanGrid] = grid;
        e[kPlanSeqs] = S;
        if (c >= G)
            continue;
        const long long s_c = c * total / G, e_c = (c + 1) * total / G;
        int s;
        long long base;
        if (ps.unit_major) {
            // unit u of every sequence is a row of Wrow positions
            const long long u = s_c / Wrow, inner = s_c - u * Wrow;
            s = (int)(std::upper_bound(cum.begin(), cum.end(), inner) - cum.begin()) - 1;
            base = u * Wrow + cum[s];
        } else {
            s = (int)(std::upper_bound(start.begin(), start.end(), s_c) - start.begin()) - 1;
            base = start[s];
        }
        if (s < 0 || s >= S)
            continue;
        e[kPlanSeq] = s;
        put64(e, kPlanBase, base);
        e[kPlanLen] = ps.len[s];
        e[kPlanAux] = ps.aux[s];
        put64(e, kPlanStart, s_c);
        put64(e, kPlanEnd, e_c);
        // the first item's first block, when it is in the unit holding s_c
        const long long a =
            ps.unit_major ? base : base + (s_c > base ? (s_c - base) / span[s] : 0) * span[s];
        const long long ra = a + kUnitCost;
        const long long into = std::max(ra, s_c) - ra;
        const int j0 = ps.first[s] + (int)std::min<long long>(into * bps, ps.nb[s] - ps.first[s]);
        e[kPlanJ0] = j0;
        for (int k = 0; k < kPlanWindow; ++k) {
            const int j = j0 + k;
            e[kPlanBlocks + k] = j < W ? block_tables[(size_t)s * W + j] : -1;
        }
    }
}

// Persistent grid of one shared-prefix launch (pass 1 or 0) on the current device,
// planned (0: cannot launch or no device).
int plan_grid_shared(pa_dtype dtype, int num_q_heads, int num_kv_heads, int head_dim,
                     int block_size, int pass)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    const int sms = sm_count(dev);
    if (sms <= 0)
        return 0;
    static const int32_t kSelect = 0;  // any non-null share / plan selects the instance
    DecodeLaunch L;
    std::memset(&L, 0, sizeof L);
    L.p.plan = &kSelect;
    L.p.share = &kSelect;
    L.p.pass = pass;
    L.p.balanced = 1;
    L.p.num_q_heads = num_q_heads;
    L.p.num_kv_heads = num_kv_heads;
    L.p.group = num_q_heads / num_kv_heads;
    L.p.head_groups = (L.p.group + kHeadsPerItem - 1) / kHeadsPerItem;
    L.head_dim = head_dim;
    L.block_size = block_size;
    L.sm_count = sms;
    L.grid = 0;
    return dtype == PA_F32 ? plan_grid_f32(L) : dtype == PA_F16 ? plan_grid_f16(L) : plan_grid_bf16(L);
}

bool shared_plan_args_ok(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                         int block_size, int max_blocks_per_seq, int dtype)
{
    return plan_args_ok(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                        max_blocks_per_seq, dtype) &&
           num_q_heads / num_kv_heads <= kHeadsPerItem;
}

}  // namespace

extern "C" {

size_t pa_decode_shared_plan_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, int max_blocks_per_seq, pa_dtype dtype)
{
    if (!shared_plan_args_ok(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                             max_blocks_per_seq, dtype))
        return (size_t)-1;
    const int g1 = plan_grid_shared(dtype, num_q_heads, num_kv_heads, head_dim, block_size, 1);
    const int g0 = plan_grid_shared(dtype, num_q_heads, num_kv_heads, head_dim, block_size, 0);
    if (g1 <= 0 || g1 != g0)
        return (size_t)-1;
    return 2 * (size_t)g1 * kPlanInts * sizeof(int32_t);
}

pa_status pa_decode_shared_plan(int32_t *plan, size_t plan_bytes, const int32_t *block_tables,
                                int max_blocks_per_seq, const int32_t *context_lens,
                                const int32_t *share, int num_seqs, int num_q_heads,
                                int num_kv_heads, int head_dim, int block_size, pa_dtype dtype)
{
    if (!plan || (num_seqs > 0 && (!block_tables || !context_lens || !share)))
        return PA_ERR_INVALID;
    if (!shared_plan_args_ok(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                             max_blocks_per_seq, dtype))
        return PA_ERR_INVALID;
    // both launches' entries for the same persistent grid: the plan's size gives it
    const size_t entry = (size_t)kPlanInts * sizeof(int32_t);
    if (plan_bytes == 0 || plan_bytes % (2 * entry) != 0 || plan_bytes / (2 * entry) > (1u << 20))
        return PA_ERR_INVALID;
    const int grid = (int)(plan_bytes / (2 * entry));
    const int S = num_seqs, W = max_blocks_per_seq, B = block_size;
    const int group = num_q_heads / num_kv_heads;
    const int U = num_kv_heads * ((group + kHeadsPerItem - 1) / kHeadsPerItem);
    const int bps = blocks_per_stage(dtype == PA_F32 ? 4 : 2, B);
    const int mpi = (group <= 8 ? 8 : kHeadsPerItem) / group;  // members per pass-1 item
    // each sequence's entries as the kernel reads them (seq_units)
    std::vector<int> len((size_t)S), lead((size_t)S), shared((size_t)S);
    for (int s = 0; s < S; ++s) {
        const long long t = context_lens[s];
        len[s] = (int)std::min<long long>(std::max<long long>(t, 0), (long long)W * B);
        lead[s] = share[2 * s];
        const int sp = share[2 * s + 1];
        shared[s] = (lead[s] >= 0 && sp > 0) ? std::min(sp, W) : 0;
    }
    PassStream p1, p0;
    for (PassStream *ps : {&p1, &p0}) {
        ps->n.assign((size_t)S, 0);
        ps->ns.assign((size_t)S, 0);
        ps->first.assign((size_t)S, 0);
        ps->nb.assign((size_t)S, 0);
        ps->len.assign((size_t)S, 0);
        ps->aux.assign((size_t)S, 0);
    }
    // pass 1: a group's first member streams its shared blocks once per kv head
    // and member group of up to mpi members
    for (int s = 0; s < S; ++s) {
        if (lead[s] != s || shared[s] <= 0)
            continue;
        int m = 1;
        while (s + m < S && lead[s + m] == s)
            ++m;
        p1.n[s] = num_kv_heads * ((m + mpi - 1) / mpi);
        p1.ns[s] = (shared[s] + bps - 1) / bps;
        p1.nb[s] = shared[s];
        p1.len[s] = shared[s];  // pass 1: the group's shared blocks
        p1.aux[s] = m;
    }
    // pass 0: every sequence's own blocks, after its group's shared ones
    bool prefix = false;
    for (int s = 0; s < S; ++s) {
        const int nb = (len[s] + B - 1) / B;
        int P = std::min(shared[s], nb);
        int flags = 0;
        if (P > 0 && len[s] <= shared[s] * B) {
            P = 0;  // ends inside the shared blocks: decoded alone, flagged
            flags |= kAuxShareErr;
        }
        p0.n[s] = U;
        p0.ns[s] = (nb - P + bps - 1) / bps;
        p0.first[s] = P;
        p0.nb[s] = nb;
        p0.len[s] = len[s];
        p0.aux[s] = P | flags;
        prefix |= P > 0;
    }
    p0.unit_major = prefix;
    if (prefix)
        for (int s = 0; s < S; ++s)
            p0.aux[s] |= kAuxUnitMajor;
    fill_pass_plan(plan, grid, p1, block_tables, W, bps);
    fill_pass_plan(plan + (size_t)grid * kPlanInts, grid, p0, block_tables, W, bps);
    return PA_OK;
}

pa_status pa_decode_shared_planned(void *out, const void *q, void *k_cache, void *v_cache,
                                   const void *k_new, const void *v_new,
                                   const int32_t *block_tables, int max_blocks_per_seq,
                                   const int32_t *context_lens, const int32_t *share, int num_seqs,
                                   int num_blocks, float scale, int num_q_heads, int num_kv_heads,
                                   int head_dim, int block_size, pa_dtype dtype,
                                   const int32_t *plan, size_t plan_bytes, void *workspace,
                                   size_t workspace_bytes, void *stream)
{
    if (num_seqs == 0)
        return PA_OK;
    if (!plan || !aligned(plan, 16))
        return PA_ERR_INVALID;
    const size_t need = pa_decode_shared_plan_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                    block_size, max_blocks_per_seq, dtype);
    if (need == (size_t)-1) {
        const bool unsupported =
            !dtype_ok(dtype) || (head_dim != 64 && head_dim != 128) ||
            (block_size != 16 && block_size != 32) ||
            (num_kv_heads > 0 && num_q_heads / num_kv_heads > kHeadsPerItem);
        return unsupported ? PA_ERR_UNSUPPORTED : PA_ERR_INVALID;
    }
    if (plan_bytes != need)
        return PA_ERR_INVALID;
    if (!share || !aligned(share, 8))
        return PA_ERR_INVALID;
    if ((k_new == nullptr) != (v_new == nullptr) ||
        (k_new && (!aligned(k_new, 16) || !aligned(v_new, 16))))
        return PA_ERR_INVALID;
    return decode_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                       num_seqs, num_blocks, scale, num_q_heads, num_kv_heads, head_dim, block_size,
                       dtype, 0, workspace, workspace_bytes, k_new, v_new, stream, share, plan,
                       (int)(plan_bytes / (2 * kPlanInts * sizeof(int32_t))));
}

size_t pa_decode_shared_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                       int head_dim, int block_size, int max_blocks_per_seq)
{
    const size_t base = pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                 block_size, max_blocks_per_seq, 0);
    if (base == (size_t)-1)
        return base;
    return 2 * base + prefix_buffer_bytes(num_seqs, num_q_heads, head_dim);
}

pa_status pa_decode_shared(void *out, const void *q, void *k_cache, void *v_cache,
                           const void *k_new, const void *v_new, const int32_t *block_tables,
                           int max_blocks_per_seq, const int32_t *context_lens,
                           const int32_t *share, int num_seqs, int num_blocks, float scale,
                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           pa_dtype dtype, void *workspace, size_t workspace_bytes, void *stream)
{
    if (num_seqs != 0 && (!share || !aligned(share, 8)))
        return PA_ERR_INVALID;
    if (num_seqs != 0 && ((k_new == nullptr) != (v_new == nullptr) ||
                          (k_new && (!aligned(k_new, 16) || !aligned(v_new, 16)))))
        return PA_ERR_INVALID;
    if (num_kv_heads > 0 && num_q_heads / num_kv_heads > kHeadsPerItem)
        return PA_ERR_UNSUPPORTED;
    return decode_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                       num_seqs, num_blocks, scale, num_q_heads, num_kv_heads, head_dim, block_size,
                       dtype, 0, workspace, workspace_bytes, k_new, v_new, stream, share);
}

pa_status pa_reshape_and_cache(const void *k, const void *v, void *k_cache, void *v_cache,
                               const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                               int head_dim, int block_size, int num_blocks, pa_dtype dtype,
                               void *stream)
{
    if (num_tokens == 0)
        return PA_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping)
        return PA_ERR_INVALID;
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
        return PA_ERR_INVALID;
    if (!dtype_ok(dtype))
        return PA_ERR_UNSUPPORTED;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(slot_mapping, 8))
        return PA_ERR_INVALID;
    const size_t row = (size_t)num_kv_heads * head_dim * elem_size(dtype);
    if (row % 16 != 0)
        return PA_ERR_UNSUPPORTED;
    const cudaError_t e = launch_reshape_and_cache(
        k, v, k_cache, v_cache, slot_mapping, num_tokens, row,
        (long long)num_blocks * block_size, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_copy_blocks(void *k_cache, void *v_cache, const int32_t *src_dst_pairs,
                         int num_pairs, int num_blocks, size_t block_bytes, void *stream)
{
    if (num_pairs == 0)
        return PA_OK;
    if (!k_cache || !v_cache || !src_dst_pairs || num_pairs < 0 || num_blocks <= 0 ||
        block_bytes == 0 || block_bytes % 16 != 0)
        return PA_ERR_INVALID;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(src_dst_pairs, 4))
        return PA_ERR_INVALID;
    if (block_bytes / 16 > 65535ull * 1024ull)
        return PA_ERR_UNSUPPORTED;
    const cudaError_t e = launch_copy_blocks(k_cache, v_cache, src_dst_pairs, num_pairs, num_blocks,
                                             block_bytes, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

namespace {
// A pointer the kernels may dereference: device memory, managed memory, or pinned
// host memory whose device address is the host address (unified addressing).
bool device_accessible(const void *ptr)
{
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged)
        return true;
    return at.type == cudaMemoryTypeHost && at.devicePointer == ptr;
}

bool all_accessible(std::initializer_list<const void *> ptrs)
{
    for (const void *p : ptrs)
        if (!device_accessible(p))
            return false;
    return true;
}
}  // namespace

pa_status pa_swap_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                         const int32_t *src_dst_pairs, int num_pairs, int src_num_blocks,
                         int dst_num_blocks, size_t block_bytes, void *stream)
{
    if (num_pairs == 0)
        return PA_OK;
    if (!src_k || !src_v || !dst_k || !dst_v || !src_dst_pairs || num_pairs < 0 ||
        src_num_blocks <= 0 || dst_num_blocks <= 0 || block_bytes == 0 || block_bytes % 16 != 0)
        return PA_ERR_INVALID;
    if (!aligned(src_k, 16) || !aligned(src_v, 16) || !aligned(dst_k, 16) || !aligned(dst_v, 16) ||
        !aligned(src_dst_pairs, 4))
        return PA_ERR_INVALID;
    if (block_bytes / 16 > 65535ull * 1024ull)
        return PA_ERR_UNSUPPORTED;
    if (!all_accessible({src_k, src_v, dst_k, dst_v, src_dst_pairs}))
        return PA_ERR_INVALID;
    const cudaError_t e = launch_move_blocks(src_k, src_v, dst_k, dst_v, src_dst_pairs, 2,
                                             src_dst_pairs + 1, 2, num_pairs, src_num_blocks,
                                             dst_num_blocks, block_bytes,
                                             static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

namespace {
pa_status stage_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                       const int32_t *block_ids, int num_ids, int num_blocks, size_t block_bytes,
                       bool gather, void *stream)
{
    if (num_ids == 0)
        return PA_OK;
    if (!src_k || !src_v || !dst_k || !dst_v || !block_ids || num_ids < 0 || num_blocks <= 0 ||
        block_bytes == 0 || block_bytes % 16 != 0)
        return PA_ERR_INVALID;
    if (!aligned(src_k, 16) || !aligned(src_v, 16) || !aligned(dst_k, 16) || !aligned(dst_v, 16) ||
        !aligned(block_ids, 4))
        return PA_ERR_INVALID;
    if (block_bytes / 16 > 65535ull * 1024ull)
        return PA_ERR_UNSUPPORTED;
    if (!all_accessible({src_k, src_v, dst_k, dst_v, block_ids}))
        return PA_ERR_INVALID;
    const cudaError_t e =
        gather ? launch_move_blocks(src_k, src_v, dst_k, dst_v, block_ids, 1, nullptr, 0, num_ids,
                                    num_blocks, num_ids, block_bytes,
                                    static_cast<cudaStream_t>(stream))
               : launch_move_blocks(src_k, src_v, dst_k, dst_v, nullptr, 0, block_ids, 1, num_ids,
                                    num_ids, num_blocks, block_bytes,
                                    static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}
}  // namespace

pa_status pa_gather_blocks(const void *k_cache, const void *v_cache, const int32_t *block_ids,
                           int num_ids, int num_blocks, void *staging_k, void *staging_v,
                           size_t block_bytes, void *stream)
{
    return stage_blocks(k_cache, v_cache, staging_k, staging_v, block_ids, num_ids, num_blocks,
                        block_bytes, true, stream);
}

pa_status pa_scatter_blocks(const void *staging_k, const void *staging_v, void *k_cache,
                            void *v_cache, const int32_t *block_ids, int num_ids, int num_blocks,
                            size_t block_bytes, void *stream)
{
    return stage_blocks(staging_k, staging_v, k_cache, v_cache, block_ids, num_ids, num_blocks,
                        block_bytes, false, stream);
}

int pa_kv_transfer_worthwhile(long long reusable_tokens, long long threshold_tokens)
{
    return reusable_tokens > 0 && reusable_tokens >= threshold_tokens ? 1 : 0;
}

pa_status pa_device_errors(unsigned int *flags, void *stream)
{
    if (!flags)
        return PA_ERR_INVALID;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e);
    unsigned int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_device_errors, sizeof v);
    if (e != cudaSuccess)
        return cuda_fail(e);
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_device_errors, &zero, sizeof zero);
    if (e != cudaSuccess)
        return cuda_fail(e);
    *flags = v;
    if (v & (PA_DEVERR_TIMEOUT_FULL | PA_DEVERR_TIMEOUT_EMPTY))
        return PA_ERR_TIMEOUT;
    return (v & (PA_DEVERR_SHARE | PA_DEVERR_PLAN)) ? PA_ERR_INVALID : PA_OK;
}

unsigned long long pa_set_wait_limit_ns(unsigned long long ns)
{
    return g_wait_limit_ns.exchange(ns == 0 ? kWaitTimeoutNs : ns);
}

}  // extern "C"
