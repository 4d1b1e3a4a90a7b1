// sort_noalloc.cu -- lsh_bucket_sort_noalloc: the stable bucket sort for callers that
// cannot allocate device memory.
//
// Some callers cannot hand this library a workspace: code running inside a framework
// whose allocator they do not control, plugins and inference runtimes that forbid
// allocation after start-up, and programs that must not call cudaMalloc (it can
// synchronise the device, and it can fail at a point where the caller has no way to
// recover).  This entry point runs the same three sort kernels as lsh_bucket_sort, but
// takes their scratch (the per-tile bucket counts, turned into offsets in place) from
// a fixed array compiled into the library instead of from a caller workspace.
//
// Facts a caller must know:
//  - The array holds kNoAllocScratchBytes (8 MiB).  Every GPU that loads the library
//    keeps it until the process exits.  A problem needs
//    4 * B*H*n_rounds * n_buckets * ceil(L / 4096) bytes; larger problems are
//    rejected with LSH_ERR_WORKSPACE_TOO_SMALL before anything is launched.
//  - All calls on one device share the array.  Calls that overlap on the GPU (on
//    different streams, or from different host threads without ordering) race on it
//    and corrupt each other's results; order them on one stream or serialise them.
//  - The array keeps the previous call's contents.  Nothing needs clearing: the count
//    kernel writes every entry the later kernels read.
//  - The first call on a device looks up the array's device address
//    (cudaGetSymbolAddress) with that device current; make that first call before any
//    stream capture, with the device that owns `stream` current.  The address is
//    cached for the life of the process, so after cudaDeviceReset (or any teardown of
//    the device's primary context) this entry point must not be called again on that
//    device: the cached address would no longer belong to a live allocation.
//  - No cudaMalloc, cudaFree or other allocating routine is called.
#include <mutex>

#include "internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = 8u << 20;
constexpr int kMaxDevices = 64;

// The scratch itself: one copy per device, for the life of the process.
static __device__ __align__(256) int32_t g_sort_scratch[kNoAllocScratchBytes / sizeof(int32_t)];

std::mutex g_mutex;
int32_t *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_sort_scratch on the current device (looked up once per device).
// In host code the symbol is only a host-side stand-in; its device address must come
// from cudaGetSymbolAddress.
cudaError_t scratch_for_current_device(int32_t **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_sort_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = (int32_t *)p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" lsh_status_t lsh_bucket_sort_noalloc(const int32_t *buckets, int B, int H, int L,
                                                int n_buckets, int n_rounds, int32_t *perm,
                                                int32_t *inv, int32_t *bstart, void *stream)
{
    if (B <= 0 || H <= 0 || L <= 0 || n_buckets <= 0 || n_rounds <= 0) return LSH_ERR_INVALID_ARGUMENT;
    if (!buckets || !perm || !inv || !bstart) return LSH_ERR_INVALID_ARGUMENT;
    if (n_buckets > 2048) return LSH_ERR_UNSUPPORTED;
    if ((long long)B * H * n_rounds * L >= (1LL << 31)) return LSH_ERR_UNSUPPORTED;
    const unsigned long long need =
        4ull * B * H * n_rounds * (unsigned long long)n_buckets * lsh::sort_tiles(L);
    if (need > kNoAllocScratchBytes) return LSH_ERR_WORKSPACE_TOO_SMALL;
    int32_t *scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return LSH_ERR_CUDA;
    lsh::Problem p;
    p.B = B; p.H = H; p.L = L; p.d = 64; p.nb = n_buckets; p.n_rounds = n_rounds;
    p.chunk = 32; p.causal = 0; p.scale = 1.f; p.dtype = LSH_F32;
    const cudaError_t e = lsh::sort_launch(p, buckets, perm, inv, bstart, scratch,
                                           (cudaStream_t)stream);
    return e == cudaSuccess ? LSH_OK : LSH_ERR_CUDA;
}
