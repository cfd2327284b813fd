// noalloc.cu -- usp_forward for callers that cannot allocate device memory themselves.
//
// The workspace of usp_forward normally comes from the caller. Some callers have no way to provide
// one: a plugin living inside a host application whose memory manager owns every device byte (a
// serving engine that reserves the GPU up front and forbids allocations outside its pool), or a
// caller on a latency-critical path that must not pay for cudaMalloc / cudaFree, which can
// synchronise the device. This variant takes its workspace from a fixed array that belongs to this
// library instead, so the call itself allocates nothing.
#include <mutex>

#include "usp_internal.cuh"

// The scratch: one file-scope device array, present on every GPU that loads this library until the
// process exits. Every call on a device uses the same array and leaves its contents behind; nothing
// in it has to start at zero (usp_forward writes every workspace byte before reading it).
static __device__ __align__(256) unsigned char g_usp_noalloc_scratch[USP_NOALLOC_SCRATCH_BYTES];

namespace usp {
namespace {

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch on the current device. Host code cannot use the array's name as a
// device address (it is a host-side stand-in), so the address is looked up once per device, with
// that device current, and cached.
void *scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_usp_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch_addr[dev] = p;
    }
    return g_scratch_addr[dev];
}

}  // namespace
}  // namespace usp

extern "C" {

int usp_forward_noalloc(const void *q, const void *k, const void *v, void *out, float *lse, usp_attn_desc d,
                        int head_chunk, usp_stream_t stream) {
    const size_t need = usp_forward_workspace_size(d, head_chunk, 0);
    // invalid arguments (or nothing to do): usp_forward reports the exact status before any launch
    if (need == 0) return usp_forward(q, k, v, out, lse, d, head_chunk, nullptr, 0, stream);
    if (need > (size_t)USP_NOALLOC_SCRATCH_BYTES) return USP_ERR_UNSUPPORTED;
    // the sequence must split into 2 rd equal chunks and L / rd into ud parts; checked here, before the
    // first touch of the device
    if (d.L % (2 * (int64_t)d.rd) != 0 || (d.L / d.rd) % d.ud != 0) return USP_ERR_SHAPE;
    void *ws = usp::scratch_address();
    if (!ws) return USP_ERR_CUDA;
    return usp_forward(q, k, v, out, lse, d, head_chunk, ws, (size_t)USP_NOALLOC_SCRATCH_BYTES, stream);
}

}  // extern "C"
