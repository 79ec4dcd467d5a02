// pe_linear_noalloc: the plain GEMM entry point for callers that cannot
// allocate device memory.
//
// Some callers must not call cudaMalloc at the point where they run a GEMM:
// code that executes while another thread captures a CUDA graph in global
// capture mode (where cudaMalloc is prohibited), and runtimes whose device
// memory is entirely reserved up front by their own allocator. pe_linear
// asks such callers for split-K scratch; this variant instead keeps that
// scratch in fixed arrays compiled into the library, so a call allocates
// nothing. The arrays exist once per device that loads the library and stay
// until the process exits.
#include <mutex>
#include <string>

#include "common.cuh"
#include "internal.h"

namespace {

constexpr size_t kWsFloats = static_cast<size_t>(2) << 20;   // 2 Mi floats = 8 MiB of split-K partials
constexpr int kTickets = 4096;                               // per-tile arrival counters

static __device__ __align__(256) float g_ws[kWsFloats];
static __device__ __align__(256) int g_tickets[kTickets];

struct DeviceScratch {
    float* ws = nullptr;
    int* tickets = nullptr;
};
std::mutex g_mutex;
DeviceScratch g_scratch[64];

// Device addresses of the arrays on the current device. In host code the
// array names are host-side stand-ins, so the addresses come from
// cudaGetSymbolAddress, looked up once per device with that device current.
// The cached addresses stay valid for the life of the device's primary
// context: after cudaDeviceReset the library must not be called on that
// device again in this process.
int scratch_for_current_device(DeviceScratch* out) {
    int dev = 0;
    PE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) {
        pe::set_error("pe_linear_noalloc: device ordinal out of range");
        return PE_ERR_ARG;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceScratch& s = g_scratch[dev];
    if (s.ws == nullptr) {
        void* ws = nullptr;
        void* tk = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ws, g_ws);
        if (e != cudaSuccess) {
            pe::set_error(std::string("pe_linear_noalloc: cudaGetSymbolAddress(scratch): ") + cudaGetErrorString(e));
            return PE_ERR_CUDA;
        }
        e = cudaGetSymbolAddress(&tk, g_tickets);
        if (e != cudaSuccess) {
            pe::set_error(std::string("pe_linear_noalloc: cudaGetSymbolAddress(tickets): ") + cudaGetErrorString(e));
            return PE_ERR_CUDA;
        }
        // both dtype instances of the kernel, so that a first call in the
        // other dtype later loads no module
        const int rc = pe::gemm_store_kernels_load();
        if (rc != PE_OK) return rc;
        s.ws = static_cast<float*>(ws);
        s.tickets = static_cast<int*>(tk);
    }
    *out = s;
    return PE_OK;
}

}  // namespace

using namespace pe;

extern "C" int pe_linear_noalloc(int32_t dtype, int32_t M, int32_t N, int32_t Kd, const void* w, const void* x,
                                 float* y, void* stream) {
    if (!w || !x || !y) { set_error("null tensor argument"); return PE_ERR_ARG; }
    if (dtype != PE_DTYPE_BF16 && dtype != PE_DTYPE_FP32) { set_error("unknown dtype"); return PE_ERR_ARG; }
    if (M < 1 || N < 1 || Kd < 1 || Kd % 8 != 0) {
        set_error("need M, N >= 1 and Kd a positive multiple of 8");
        return PE_ERR_ARG;
    }
    int dev = 0, sms = 0;
    PE_CUDA_TRY(cudaGetDevice(&dev));
    PE_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    const int eb = dtype == PE_DTYPE_BF16 ? 2 : 4;
    const GemmPlan g = plan_gemm(M, N, Kd, EPI_STORE, eb, sms, false);
    // the tickets are used only by split-K plans (one per tile)
    if (g.ws_floats > kWsFloats || (g.splits > 1 && g.tiles > kTickets)) {
        set_error("pe_linear_noalloc: this shape needs " + std::to_string(g.ws_floats) + " floats of split-K scratch and " +
                  std::to_string(g.tiles) + " tickets; the built-in maximum is " + std::to_string(kWsFloats) +
                  " floats and " + std::to_string(kTickets) + " tickets (use pe_linear)");
        return PE_ERR_ARG;
    }
    DeviceScratch sc;
    int rc = scratch_for_current_device(&sc);
    if (rc != PE_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // Tickets must be zero when the kernel starts. A completed call leaves
    // them zero; clearing them on the stream also covers a call that was
    // interrupted. The partials need no clearing: every split writes its
    // whole tile before any split reads it.
    if (g.splits > 1) PE_CUDA_TRY(cudaMemsetAsync(sc.tickets, 0, static_cast<size_t>(g.tiles) * sizeof(int), s));
    CUtensorMap ta, tb;
    rc = encode_tmap_2d(&ta, w, dtype, Kd, M, static_cast<uint64_t>(Kd) * eb, 128 / eb, 128);
    if (rc == PE_OK) rc = encode_tmap_2d(&tb, x, dtype, Kd, N, static_cast<uint64_t>(Kd) * eb, 128 / eb, g.bn);
    if (rc != PE_OK) return rc;
    GemmParams p{};
    p.M = M;
    p.N = N;
    p.Kd = Kd;
    p.out_f32 = y;
    p.ld_out = M;
    p.ws = sc.ws;
    p.tickets = sc.tickets;
    p.err = nullptr;
    return launch_gemm(dtype, EPI_STORE, ta, ta, tb, g, p, s, false);
}
