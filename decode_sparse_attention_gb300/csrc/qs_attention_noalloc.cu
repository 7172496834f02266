// Sparse decode attention for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: code that runs
// where a device allocation is not allowed or not available (an inference
// engine's decode loop that forbids allocations after warm-up, a plugin that
// receives only input and output pointers from its host framework, an
// embedded runtime without a device allocator).  This entry point runs the
// same split-K attention kernel with its scratch (the per-unit arrival
// counters and the split-K partial results) taken from a fixed array that the
// library itself carries in device memory.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it until the process exits.  Host code cannot pass the
// array's name to a kernel (on the host that name is only a stand-in), so the
// first call on each device looks up the array's device address with
// cudaGetSymbolAddress while that device is current, and later calls on the
// device reuse the address.  Because of that look-up, make the first call on
// a device outside of any stream capture.
//
// Every call on a device uses the same array and it keeps what the previous
// call left there, so each call clears the arrival counters it is going to
// use (a memset enqueued on the caller's stream once every argument check has
// passed; a rejected call enqueues nothing).  Two calls whose work overlaps on
// the GPU -- e.g. on two streams without ordering between them -- race on the
// array and give wrong results; order such calls on one stream.  The call
// allocates nothing: no cudaMalloc, no cudaFree, no library routine that
// allocates.
#include <mutex>

#include "qs_internal.cuh"

namespace qs {

namespace {

// Maximum scratch of one call: 4 MiB.  A call needs one 4-byte arrival
// counter per unit (rounded up to 256 bytes) plus 2 * units + 1024 partial
// slots of G * (D + 2) floats (the same formula as the workspace entry
// point), so at H/N = 4, D = 128 (2080-byte slots) it serves at most 495
// (request, KV head) units; 496 units already need 4,195,328 bytes.
constexpr size_t kStaticScratchBytes = size_t(4) << 20;

__device__ __align__(256) uint8_t g_attn_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of g_attn_scratch on the current device (looked up once).
void* scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace qs

extern "C" qs_status qs_sparse_decode_attn_noalloc(
    const void* q, qs_dtype q_dtype, const void* k_cache, const void* v_cache,
    const float* k_scale, const float* v_scale, qs_dtype kv_dtype, int32_t num_kv_blocks,
    const int32_t* block_tables, int32_t MKBPR, const int32_t* seq_lens, const int32_t* selected,
    int32_t sel_heads, int32_t k, float softmax_scale, int32_t B, int32_t H, int32_t N,
    int32_t D, int32_t BS, float* out, float* lse_opt, int32_t* dev_status, qs_stream_t stream) {
    using namespace qs;
    if (B < 0 || H <= 0 || N <= 0 || H % N != 0 || D <= 0) return QS_EINVAL;
    if (sel_heads != N && sel_heads != H) return QS_EINVAL;
    if (B == 0) return QS_OK;
    const size_t need = attn_workspace_bytes(B, H, N, D, sel_heads);
    if (need > kStaticScratchBytes) return QS_EWORKSPACE;  // beyond the fixed 4 MiB scratch
    void* scratch = scratch_on_current_device();
    if (!scratch) return QS_ECUDA;
    // the arrival counters must start at zero: sparse_attn_impl clears them
    // on the stream after its checks; the partial slots are written before
    // they are read
    return sparse_attn_impl(q, q_dtype, k_cache, v_cache, k_scale, v_scale, kv_dtype,
                            num_kv_blocks, block_tables, MKBPR, seq_lens, selected, sel_heads, k,
                            softmax_scale, B, H, N, D, BS, out, lse_opt, scratch,
                            kStaticScratchBytes, dev_status, reinterpret_cast<cudaStream_t>(stream),
                            /*pdl=*/false, /*clear_counters=*/true);
}

extern "C" qs_status qs_sparse_decode_attn_noalloc_scratch(void** device_ptr, size_t* bytes) {
    if (!device_ptr || !bytes) return QS_EINVAL;
    void* p = qs::scratch_on_current_device();
    if (!p) return QS_ECUDA;
    *device_ptr = p;
    *bytes = qs::kStaticScratchBytes;
    return QS_OK;
}
