// noalloc.cu -- sdtw_forward_noalloc: the forward pass with library-owned,
// statically sized scratch, for callers that cannot allocate device memory.
//
// Who needs it: a host program that drives this library without any device
// allocator of its own (no PyTorch, no memory pool), or a loop that must not
// call into the CUDA allocator at all (cudaMalloc and cudaFree synchronize the
// device and can stall a latency-critical stream). Such a caller still passes
// its inputs and outputs; only the scratch of the forward comes from here.
//
// The scratch is one file-scope __device__ array of kStaticScratchBytes. Every
// GPU that loads this library holds it until the process exits. Host code
// cannot pass the array's name to a kernel (on the host the name is only a
// stand-in, not a device address), so the first call on each device, with that
// device current, looks up the device address once with cudaGetSymbolAddress
// and caches it; that first call should come before any stream capture.
// All calls share the array and it keeps the last call's contents: the control
// words that must start at zero are cleared at the start of every call (an
// asynchronous memset on the caller's stream), and calls that overlap on the
// GPU (different streams, or several host threads) race on it. The cached
// address belongs to the device's current context: after cudaDeviceReset the
// module is loaded again and the array may move, so the cache is not valid
// across a reset. A device-side wait that runs out of time leaves NaN in every
// loss of the call (there is no workspace whose status word the caller could
// read).
#include <cstdint>
#include <mutex>

#include "../../include/sdtw.h"
#include "common.cuh"
#include "kernels.h"

using namespace sdtw;

namespace {

constexpr size_t kStaticScratchBytes = 64ull << 20;  // 64 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

size_t up256(size_t v) { return (v + 255) & ~(size_t)255; }

// loss[b] = NaN for every b when the status word reports a timed-out wait.
__global__ void poison_on_status_kernel(const int* status, float* loss, int B)
{
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B && *status != 0) loss[b] = __int_as_float(0x7fc00000);
}

// Forward-only carve of the scratch: status, control words, loss partials, last
// row, strip boundary rows, the (vl,hu) pairs and, unfused, the cost tensor.
struct FwdCarve {
    size_t status, ctrl, ctrl_bytes, colsum, rowbuf, edge, vh, dsk, total;
};

FwdCarve carve(int B, int N, int M, bool fused)
{
    const int NB = (N + 31) / 32;
    const size_t slots = (size_t)skew_slots(N, M) * B;
    FwdCarve c{};
    size_t o = 0;
    c.status = o; o = up256(o + sizeof(int));
    c.ctrl = o; c.ctrl_bytes = sizeof(int) * (1 + (size_t)B); o = up256(o + c.ctrl_bytes);
    c.colsum = o; o = up256(o + sizeof(double) * (size_t)B * NB);
    c.rowbuf = o; o = up256(o + sizeof(float) * (size_t)B * M);
    c.edge = o; o = up256(o + sizeof(Slot) * (size_t)B * NB * M);
    c.vh = o; o = up256(o + sizeof(float2) * slots);
    c.dsk = o; if (!fused) o = up256(o + sizeof(float) * slots);
    c.total = o;
    return c;
}

// Device address of the static scratch on the current device (set up once per device).
sdtw_status scratch_for_current_device(void** addr, int* sms)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SDTW_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return SDTW_ERR_CUDA;
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        g_scratch_addr[dev] = p;
        g_num_sms[dev] = n;
    }
    *addr = g_scratch_addr[dev];
    *sms = g_num_sms[dev];
    return SDTW_OK;
}

}  // namespace

extern "C" sdtw_status sdtw_forward_noalloc(const float* x, const float* y, int B, int N, int M, int D,
                                            float gamma, sdtw_mode mode, float* loss, void* stream)
{
    if (B < 1 || N < 1 || M < 1 || D < 1) return SDTW_ERR_EMPTY;
    if (!(gamma > 0.f) || !(gamma < 3.0e38f)) return SDTW_ERR_GAMMA;
    if (mode != SDTW_UNFUSED && mode != SDTW_FUSED) return SDTW_ERR_ARG;
    if (!x || !y || !loss) return SDTW_ERR_ARG;
    if (B > 65535 || N > (1 << 24) || M > (1 << 24) || D > 400) return SDTW_ERR_TOO_LARGE;
    const bool fused = (mode == SDTW_FUSED);
    if (fused && wave_smem_fixed(1, false) + wave_smem_fused_per_warp(D) > 220 * 1024) return SDTW_ERR_TOO_LARGE;
    if ((long long)N * M > (1ll << 40)) return SDTW_ERR_TOO_LARGE;
    const FwdCarve c = carve(B, N, M, fused);
    if (c.total > kStaticScratchBytes) return SDTW_ERR_TOO_LARGE;  // beyond the static scratch

    void* base = nullptr;
    int sms = 0;
    sdtw_status s = scratch_for_current_device(&base, &sms);
    if (s != SDTW_OK) return s;
    char* ws = static_cast<char*>(base);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // Warps per CTA: about one 32-row block per SM over the batch, within the
    // shared memory a fused CTA needs.
    const int NB = (N + 31) / 32;
    int W = (int)(((long long)B * NB + sms - 1) / sms);
    if (W > NB) W = NB;
    if (W > kMaxWarps) W = kMaxWarps;
    if (W < 1) W = 1;
    if (fused) {
        if (W > 8) W = 8;
        while (W > 1 && wave_smem_fixed(W, false) + (size_t)W * wave_smem_fused_per_warp(D) > 220 * 1024) --W;
    }

    Problems pr{};
    pr.xs[0] = x;
    pr.ys[0] = y;
    pr.xstride[0] = (long long)N * D;
    pr.ystride[0] = (long long)M * D;
    pr.B = B;

    WaveParams q{};
    q.pr = pr;
    q.P = B; q.N = N; q.M = M; q.D = D; q.NB = NB;
    q.W = W;
    q.S = (NB + W - 1) / W;
    q.scale = (float)(1.4426950408889634 / (double)gamma);
    q.unscale = (float)((double)gamma * 0.6931471805599453);
    q.Dsk = fused ? nullptr : reinterpret_cast<const float*>(ws + c.dsk);
    q.VH = reinterpret_cast<float2*>(ws + c.vh);
    q.E = nullptr;
    q.edge_f = reinterpret_cast<Slot*>(ws + c.edge);
    q.edge_b = nullptr;
    int* ctrl = reinterpret_cast<int*>(ws + c.ctrl);
    q.ticket_f = ctrl;
    q.done = ctrl + 1;
    q.ticket_b = nullptr;
    q.colsum = reinterpret_cast<double*>(ws + c.colsum);
    q.rowsum = nullptr;
    q.rowbuf = reinterpret_cast<float*>(ws + c.rowbuf);
    q.loss = loss;
    q.status = reinterpret_cast<int*>(ws + c.status);
    q.wait_ns = debug_wait_ns();
    q.skip_publish = debug_take_skip_publish();

    // The status word, the ticket, the counters and the strip boundary slots start at zero.
    if (cudaMemsetAsync(ws + c.status, 0, sizeof(int), st) != cudaSuccess) return SDTW_ERR_CUDA;
    if (cudaMemsetAsync(ws + c.ctrl, 0, c.ctrl_bytes, st) != cudaSuccess) return SDTW_ERR_CUDA;
    if (q.S > 1 && cudaMemsetAsync(ws + c.edge, 0, sizeof(Slot) * (size_t)B * q.S * M, st) != cudaSuccess)
        return SDTW_ERR_CUDA;
    if (!fused && launch_dist_skewed(pr, B, N, M, D, reinterpret_cast<float*>(ws + c.dsk), st) != cudaSuccess)
        return SDTW_ERR_CUDA;
    if (launch_forward(q, fused, st) != cudaSuccess) return SDTW_ERR_CUDA;
    // a wait that ran out of time makes every loss of the call NaN
    poison_on_status_kernel<<<(B + 255) / 256, 256, 0, st>>>(q.status, loss, B);
    if (cudaGetLastError() != cudaSuccess) return SDTW_ERR_CUDA;
    return SDTW_OK;
}
