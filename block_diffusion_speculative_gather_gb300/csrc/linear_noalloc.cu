// dflash_linear_noalloc: the standalone weight-streaming GEMM of
// dflash_linear for callers that cannot allocate device memory.
//
// The GEMM splits long reductions across CTAs and needs scratch for the
// partial tiles, the per-tile tickets and a small state word.  dflash_linear
// takes that scratch from a caller workspace; this entry point takes it from
// one fixed array in the library's own device memory instead, so the caller
// passes nothing but the operands.  The array exists once per GPU that loads
// the library and lives until the process exits.
//
// Limits and sharing:
//  * n (output columns) at most LINEAR_NOALLOC_MAX_N; larger n is rejected
//    with DFLASH_ERR_ARG before anything is launched;
//  * every call on a device uses the same array.  Each call clears the
//    tickets and the state words on its stream before the GEMM; the partial
//    tiles are always written before they are read.  Two calls that overlap
//    on the GPU (different streams without ordering between them) race on
//    the array and may return wrong results;
//  * the kernel's bounded waits report through the caller's err words: the
//    call copies the state's (code, site) pair there after the GEMM, so a
//    wait that ran out (y incomplete) is seen by the caller once the stream
//    reaches that point, although the call itself has returned DFLASH_OK;
//  * the array's device address is looked up once per device and kept; a
//    cudaDeviceReset (which unloads the library's module from that device)
//    invalidates it, so the entry point must not be used after one.

#include <cstring>
#include <mutex>

#include "../../include/dflash.h"
#include "gemm.cuh"

using namespace dfl;

namespace {

constexpr int LINEAR_NOALLOC_MAX_N = 262144;                  // output columns
constexpr int NOALLOC_MAX_CTAS = 256 * DFL_GEMM_CTAS_PER_SM;  // GEMM grid bound
constexpr size_t NOALLOC_SLOT_BYTES =
    (size_t)NOALLOC_MAX_CTAS * 2 * GEMM_BN * DFL_MAX_ROWS * sizeof(float);   // 4 MiB
constexpr size_t NOALLOC_TICKET_BYTES = (size_t)(LINEAR_NOALLOC_MAX_N / GEMM_BN) * sizeof(int);
constexpr size_t NOALLOC_STATE_BYTES = 1024;
static_assert(sizeof(DevState) <= NOALLOC_STATE_BYTES, "state word region too small");
constexpr size_t NOALLOC_BYTES = NOALLOC_SLOT_BYTES + NOALLOC_TICKET_BYTES + NOALLOC_STATE_BYTES;

constexpr int NOALLOC_MAX_DEVICES = 64;

}  // namespace

// The scratch itself: [partial tiles][tickets][state].  In host code this
// name is only a stand-in for the symbol; its device address comes from
// cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_linear_noalloc_scratch[NOALLOC_BYTES];

namespace {

std::mutex g_setup_mu;
unsigned char* g_scratch_addr[NOALLOC_MAX_DEVICES];   // device address per device
int g_scratch_sms[NOALLOC_MAX_DEVICES];

// Once per device, with that device current: the scratch's device address
// and the SM count that sizes the grid.
int setup_device(int dev, unsigned char** addr, int* sms) {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_linear_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return report_error(DFLASH_ERR_CUDA, "scratch address of device %d: %s", dev,
                                cudaGetErrorString(e));
        int n_sm = 0;
        e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return report_error(DFLASH_ERR_CUDA, "SM count of device %d: %s", dev,
                                cudaGetErrorString(e));
        g_scratch_sms[dev] = n_sm > 256 ? 256 : n_sm;
        g_scratch_addr[dev] = static_cast<unsigned char*>(p);
    }
    *addr = g_scratch_addr[dev];
    *sms = g_scratch_sms[dev];
    return DFLASH_OK;
}

}  // namespace

extern "C" int dflash_linear_noalloc(const void* w, const void* x, int32_t n, int32_t k, float* y,
                                     int32_t* err, dflash_stream_t stream) {
    if (!w || !x || !y || !err) return report_error(DFLASH_ERR_ARG, "NULL argument");
    if (n < GEMM_BN || n % GEMM_BN || k < 64 || k % 64)
        return report_error(DFLASH_ERR_ARG, "n %d k %d: n a multiple of 128, k of 64", n, k);
    if (n > LINEAR_NOALLOC_MAX_N)
        return report_error(DFLASH_ERR_ARG,
                            "n %d exceeds %d, the most output columns the fixed scratch serves "
                            "(use dflash_linear with a workspace)", n, LINEAR_NOALLOC_MAX_N);
    if ((reinterpret_cast<uintptr_t>(y) & 15) != 0 || (reinterpret_cast<uintptr_t>(err) & 7) != 0)
        return report_error(DFLASH_ERR_ARG, "y or err misaligned");
    const cudaError_t pending = cudaGetLastError();
    if (pending != cudaSuccess)
        return report_error(DFLASH_ERR_CUDA, "a CUDA error was pending before this call: %s",
                            cudaGetErrorString(pending));
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return report_error(DFLASH_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= NOALLOC_MAX_DEVICES)
        return report_error(DFLASH_ERR_ARG, "device %d: at most %d devices", dev, NOALLOC_MAX_DEVICES);
    unsigned char* base = nullptr;
    int sms = 0;
    const int r = setup_device(dev, &base, &sms);
    if (r) return r;
    // tickets and state start at zero on every call (an earlier call may
    // have been cut short by a wait that ran out)
    unsigned char* tickets = base + NOALLOC_SLOT_BYTES;
    return run_linear_store(w, x, n, k, y, reinterpret_cast<float*>(base),
                            reinterpret_cast<int*>(tickets),
                            reinterpret_cast<DevState*>(tickets + NOALLOC_TICKET_BYTES), tickets,
                            NOALLOC_TICKET_BYTES + NOALLOC_STATE_BYTES, err, sms,
                            reinterpret_cast<cudaStream_t>(stream));
}
