// csa2_layer_noalloc: csa2_layer without a caller-provided workspace.
//
// Some callers cannot allocate device memory per call: code that runs as a
// plugin of a host program which owns every device allocation, or a serving
// loop that forbids allocations after start-up.  For them the scratch of a
// layer lives in one static device array compiled into this library, so the
// call needs nothing but its inputs and outputs.
//
// The array is a host-side stand-in in host code; its device address is
// looked up once per device (cudaGetSymbolAddress with that device current)
// on the first call made on that device, and cached.
#include <mutex>

#include "csa2_internal.cuh"

static __device__ __align__(256) unsigned char g_noalloc_scratch[CSA2_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};
}  // namespace

extern "C" int csa2_layer_noalloc(int32_t mode, const csa2_cache *cache, const csa2_batch *batch,
                                  const csa2_layer_io *io, csa2_stream_t stream)
{
    if (!batch) return CSA2_ERR_NULL;
    // every call shares the one array, so no call can have a workspace of its own
    if (io && (io->swa.flags & CSA2_ATTN_EARLY_ALL)) return CSA2_ERR_UNSUPPORTED;
    // reject work whose scratch does not fit before touching the device
    const size_t need = csa2::layer_workspace_need(mode, batch, io);
    if (need > (size_t)CSA2_NOALLOC_SCRATCH_BYTES) return CSA2_ERR_WORKSPACE;

    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        csa2::set_cuda_error(e);
        return CSA2_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return CSA2_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_scratch_ptr[dev]) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
            if (e != cudaSuccess) {
                csa2::set_cuda_error(e);
                return CSA2_ERR_CUDA;
            }
            g_scratch_ptr[dev] = p;
        }
        scratch = g_scratch_ptr[dev];
    }
    return csa2_layer(mode, cache, batch, io, scratch, (size_t)CSA2_NOALLOC_SCRATCH_BYTES, stream);
}
