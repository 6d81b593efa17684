// api.cu -- the C ABI of libsdtw.so: validation, workspace carving, launches.
//
// Each entry point validates its arguments on the host (returning before any
// launch on error), carves the caller's workspace, and enqueues its kernels on
// the caller's stream. Nothing is allocated here.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/sdtw.h"
#include "common.cuh"
#include "kernels.h"

using namespace sdtw;

namespace {

constexpr size_t kAlign = 256;
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s

unsigned long long g_wait_ns = kDefaultWaitNs;
int g_skip_publish = 0;

// Kernel choices forced by sdtw_debug_set_options and sdtw_debug_set_clusters
// (testing only; zeros: the library's own choices).
struct DebugOptions {
    int warps_fwd, warps_bwd;   // warps per wavefront CTA (> 0: forced)
    int dist_simt, fused_simt;  // difference-form cost kernels (unfused / fused, both precisions)
    int max_cluster;            // CTAs per cluster of the fused tensor-core forward at most (0: up to 4)
};
DebugOptions g_dbg{};

size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

// Workspace layout. The status word sits at offset 0 for every op.
struct Layout {
    size_t status, ctrl_f, ctrl_f_bytes, ctrl_b, ctrl_b_bytes;
    size_t ctrl_band, ctrl_band_stride;  // checkpointed mode: each band launch's own counters
    size_t colsum, rowsum, rowbuf, losses, edge_f, edge_b, vh, e, dsk, gparts, gnorm, bimg, bimg2, total;
    size_t ximg, yimg, xnorm, ynorm;  // tensor-core cost operands (tc_cost, or xtc: digit images and row info)
    size_t band_slots;                // checkpointed mode: skewed slots of one band of every problem
    size_t ebnd;                      // extended mode: non-zero column range of E per 32-row block
    bool tc_cost;
    bool xtc;    // extended modes: exact tensor-core costs (D <= kMaxXtcD)
    bool ckpt;   // checkpointed fused mode: VH / E hold two bands, the [X | 1] image one
    int P, N, M, D, NB;
};

// Side streams and cached events (defined below, with their rules).
cudaStream_t side_stream();
cudaStream_t grad_stream();
cudaStream_t chain_stream(int k);
enum EventSlot {
    kEvBwdFork, kEvBwdJoin, kEvHostFork, kEvHostJoin, kEvNormFork, kEvNormJoin,
    kEvCkptFork, kEvCkptRec0, kEvCkptRec1, kEvCkptFree0, kEvCkptFree1, kEvCkptBwd0, kEvCkptBwd1, kEvCkptJoin,
    kEvCkptJoinChain,
    kEvSlots
};
cudaEvent_t cached_event(EventSlot slot);

// Checkpointed fused mode: bands of kBandBlocks 32-row blocks (the fused forward's
// 128-row strips). The forward keeps only each band's outgoing boundary row; the
// backward recomputes one band at a time.
constexpr int kBandBlocks = 4;

bool make_layout(int op, int B, int N, int M, int D, int mode, Layout* L)
{
    if (op < SDTW_OP_FWD_BWD || op > SDTW_OP_COST) return false;
    if (op == SDTW_OP_COST) D = 1;  // no features: the cost is given
    if (B < 1 || N < 1 || M < 1 || D < 1) return false;
    if (mode & ~7) return false;
    const bool fused = (mode & SDTW_FUSED) != 0, ext = (mode & SDTW_EXTENDED) != 0;
    const bool ckpt = (mode & SDTW_CHECKPOINT) != 0;
    if (op == SDTW_OP_COST && fused) return false;
    // checkpointing recomputes bands with the tensor-core fused forward (fp32, D <= 256)
    if (ckpt && (op != SDTW_OP_FWD_BWD || !fused || ext || D > kTcKFeat * kMaxTcKBlocks)) return false;
    const int P = (op == SDTW_OP_NORMALIZED) ? 3 * B : B;
    if (op == SDTW_OP_NORMALIZED) M = N;
    const int NB = (N + 31) / 32;
    const int SB = (NB + kBandBlocks - 1) / kBandBlocks;   // bands (checkpointed mode)
    const size_t slots = (size_t)skew_slots(N, M) * P;
    // per-cell state and E: every cell, or two bands of every problem (the band being
    // differentiated and the next one up, recomputed meanwhile)
    const size_t band_slots = (size_t)P * (NB < kBandBlocks ? NB : kBandBlocks) * skew_T(M) * 32;
    const size_t vslots = ckpt ? 2 * band_slots : slots;
    L->band_slots = band_slots;
    const size_t edge_rows = ckpt ? (size_t)SB : (size_t)NB;   // boundary rows kept per problem
    size_t o = 0;
    L->status = o; o = align_up(o + sizeof(int));
    L->ctrl_f = o; L->ctrl_f_bytes = sizeof(int) * (1 + (size_t)P); o = align_up(o + L->ctrl_f_bytes);
    L->ctrl_b = o; L->ctrl_b_bytes = sizeof(int); o = align_up(o + L->ctrl_b_bytes);
    // per band: the recompute's ticket and done counters, then the band backward's
    // ticket, all zeroed by one memset before the bands run
    L->ctrl_band_stride = align_up(sizeof(int) * (2 + (size_t)P));
    L->ctrl_band = o; if (ckpt) o = align_up(o + L->ctrl_band_stride * SB);
    L->colsum = o; o = align_up(o + sizeof(double) * (size_t)P * NB);
    L->rowsum = o; o = align_up(o + sizeof(double) * (size_t)P);
    L->rowbuf = o; o = align_up(o + sizeof(float2) * (size_t)P * M);
    L->losses = o; o = align_up(o + sizeof(float) * (size_t)P);
    L->edge_f = o; o = align_up(o + 2 * sizeof(Slot) * (size_t)P * edge_rows * M);
    L->edge_b = o; o = align_up(o + 2 * sizeof(Slot) * (size_t)P * edge_rows * M);
    L->vh = o; o = align_up(o + (ext ? sizeof(float4) : sizeof(float2)) * vslots);
    L->e = o; o = align_up(o + sizeof(float) * vslots);
    L->dsk = o; if (!fused) o = align_up(o + (ext ? sizeof(float2) : sizeof(float)) * slots);
    L->gparts = o; if (op == SDTW_OP_BARYCENTER) o = align_up(o + sizeof(float) * (size_t)P * N * D);
    L->gnorm = o; if (op == SDTW_OP_BARYCENTER) o = align_up(o + sizeof(float) * (((size_t)N * D + 255) / 256));
    L->ebnd = o; if (ext && op != SDTW_OP_COST) o = align_up(o + sizeof(int2) * (size_t)P * NB);
    // gradient operand images (one batch of B problems at a time): [Y | 1] and [X | 1]
    const bool xy = op != SDTW_OP_COST;  // the path has x and y (and input gradients)
    L->bimg = o; if (!ext && xy) o = align_up(o + egemm_bimg_bytes(op == SDTW_OP_NORMALIZED ? B : P, M, D));
    L->bimg2 = o;
    if (!ext && xy) o = align_up(o + egemm_bimg_bytes(op == SDTW_OP_NORMALIZED ? B : P, ckpt ? (N < 32 * kBandBlocks ? N : 32 * kBandBlocks) : N, D));
    // operand images and norms of the tensor-core costs (fp32 modes, D <= 256): the
    // unfused cost tensor and the fused forward's cost tiles
    L->tc_cost = !ext && D <= kTcKFeat * kMaxTcKBlocks && xy;
    // the extended modes' exact tensor-core costs (the fused forward's cost tiles, the
    // unfused cost tensor): fixed-point digit images and row info
    L->xtc = ext && xy && D <= kMaxXtcD;
    L->ximg = o; if (L->tc_cost) o = align_up(o + simg_bytes(P, N, D));
    if (L->xtc) o = align_up(o + oimg_bytes(P, N, D));
    L->yimg = o; if (L->tc_cost) o = align_up(o + simg_bytes(P, M, D));
    if (L->xtc) o = align_up(o + oimg_bytes(P, M, D));
    L->xnorm = o; if (L->tc_cost) o = align_up(o + snorm_bytes(P, N));
    if (L->xtc) o = align_up(o + oinfo_bytes(P, N));
    L->ynorm = o; if (L->tc_cost) o = align_up(o + snorm_bytes(P, M));
    if (L->xtc) o = align_up(o + oinfo_bytes(P, M));
    L->total = o;
    L->P = P; L->N = N; L->M = M; L->D = D; L->NB = NB;
    L->ckpt = ckpt;
    return true;
}

template <typename T>
T* at(void* ws, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(ws) + off); }

// Warps per wavefront CTA: about one 32-row block per SM partition over the
// whole batch, bounded by the shared memory a fused CTA needs.
int choose_warps(int P, int NB, int D, bool fused, bool ext, bool backward, int num_sms)
{
    int W = backward ? g_dbg.warps_bwd : g_dbg.warps_fwd;
    if (W <= 0) {
        const long long blocks = (long long)P * NB;
        W = (int)((blocks + num_sms - 1) / num_sms);
    }
    if (W > NB) W = NB;
    if (W > kMaxWarps) W = kMaxWarps;
    if (ext && backward && W > kMaxWarpsBwdExt) W = kMaxWarpsBwdExt;
    if (W < 1) W = 1;
    if (fused) {
        if (W > 8) W = 8;  // fused CTAs are at most 256 threads (register budget of the cost rows)
        const size_t limit = 220 * 1024;
        const size_t per = ext ? wavex_smem_fused_per_warp(D) : wave_smem_fused_per_warp(D);
        while (W > 1 && wave_smem_fixed(W, true) + (size_t)W * per > limit) --W;
    }
    return W;
}

int num_sms()
{
    static int n = 0;
    if (n == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
        n = v;
    }
    return n;
}

// SMs the batch being launched may count on: the whole device, or its share
// while the chunks of a host-buffer call run side by side on several streams.
thread_local int t_sm_share = 0;
int sm_budget() { return t_sm_share > 0 ? t_sm_share : num_sms(); }

// allow_ckpt: the entry point takes SDTW_CHECKPOINT (sdtw_forward / sdtw_backward and
// their padded-batch forms), which needs the tensor-core fused forward.
sdtw_status check_common(const void* x, const void* y, int B, int N, int M, int D, float gamma, int mode,
                         bool allow_ckpt = false)
{
    if (B < 1 || N < 1 || M < 1 || D < 1) return SDTW_ERR_EMPTY;
    if (!(gamma > 0.f) || !std::isfinite(gamma)) return SDTW_ERR_GAMMA;
    if (mode & ~(allow_ckpt ? 7 : 3)) return SDTW_ERR_ARG;
    if ((mode & SDTW_CHECKPOINT) &&
        (!(mode & SDTW_FUSED) || (mode & SDTW_EXTENDED) || D > kTcKFeat * kMaxTcKBlocks || g_dbg.fused_simt))
        return SDTW_ERR_ARG;
    if (!x || !y) return SDTW_ERR_ARG;
    if (B > 65535 / 3 || N > (1 << 24) || M > (1 << 24) || D > 400) return SDTW_ERR_TOO_LARGE;
    if ((mode & SDTW_FUSED) &&
        wave_smem_fixed(1, true) + ((mode & SDTW_EXTENDED) ? wavex_smem_fused_per_warp(D) : wave_smem_fused_per_warp(D)) >
            220 * 1024)
        return SDTW_ERR_TOO_LARGE;
    return SDTW_OK;
}

sdtw_status check_ws(void* ws, size_t ws_bytes, const Layout& L)
{
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) return SDTW_ERR_WORKSPACE;
    if (ws_bytes < L.total) return SDTW_ERR_WORKSPACE;
    return SDTW_OK;
}

WaveParams wave_params(const Problems& pr, const Layout& L, void* ws, float gamma, bool fused, bool ext, bool backward)
{
    WaveParams q{};
    q.pr = pr;
    q.P = L.P; q.N = L.N; q.M = L.M; q.D = L.D; q.NB = L.NB;
    q.W = choose_warps(L.P, L.NB, L.D, fused && !backward, ext, backward, sm_budget());
    q.S = (L.NB + q.W - 1) / q.W;
    q.C = g_dbg.max_cluster > 0 ? g_dbg.max_cluster : 4;  // a limit: the launchers pick the size
    q.scale = (float)(1.4426950408889634 / (double)gamma);
    q.unscale = (float)((double)gamma * 0.6931471805599453);
    q.Dsk = fused ? nullptr : at<float>(ws, L.dsk);
    q.VH = at<float2>(ws, L.vh);
    q.E = at<float>(ws, L.e);
    q.edge_f = at<Slot>(ws, L.edge_f);
    q.edge_b = at<Slot>(ws, L.edge_b);
    int* cf = at<int>(ws, L.ctrl_f);
    q.ticket_f = cf;
    q.done = cf + 1;
    q.ticket_b = at<int>(ws, L.ctrl_b);
    q.colsum = at<double>(ws, L.colsum);
    q.rowsum = at<double>(ws, L.rowsum);
    q.rowbuf = at<float>(ws, L.rowbuf);
    q.ext = ext ? 1 : 0;
    q.loss = at<float>(ws, L.losses);
    q.status = at<int>(ws, L.status);
    q.wait_ns = g_wait_ns;
    q.skip_publish = 0;
    return q;
}

#define SDTW_CUDA(call)                                  \
    do {                                                 \
        cudaError_t e_ = (call);                         \
        if (e_ != cudaSuccess) return SDTW_ERR_CUDA;     \
    } while (0)

// Forward over L.P problems; per-problem losses to `loss_out` (device).
// cost: when not null, the caller's (P,N,M) cost tensor replaces the distance step.
// lens_n / lens_m: per-problem lengths (device), or null for full N x M problems.
sdtw_status run_forward(const Problems& pr, const Layout& L, void* ws, float gamma, int mode, float* loss_out,
                        cudaStream_t st, const float* cost = nullptr, const int* lens_n = nullptr,
                        const int* lens_m = nullptr)
{
    const bool fused = (mode & SDTW_FUSED) != 0, ext = (mode & SDTW_EXTENDED) != 0;
    WaveParams q = wave_params(pr, L, ws, gamma, fused, ext, false);
    q.lens_n = lens_n;
    q.lens_m = lens_m;
    const bool tc = L.tc_cost && !(fused ? g_dbg.fused_simt : g_dbg.dist_simt);
    const bool xtc = L.xtc && !cost && !(fused ? g_dbg.fused_simt : g_dbg.dist_simt);
    if (fused && (tc || xtc)) {  // the tensor-core fused forwards take 128-row strips (4 warps)
        q.W = 4;
        q.S = (L.NB + 3) / 4;
    }
    SDTW_CUDA(cudaMemsetAsync(at<char>(ws, L.status), 0, sizeof(int), st));
    SDTW_CUDA(cudaMemsetAsync(at<char>(ws, L.ctrl_f), 0, L.ctrl_f_bytes, st));
    if (q.S > 1)  // strip boundary slots start untagged
        SDTW_CUDA(cudaMemsetAsync(q.edge_f, 0, (ext ? 2 : 1) * sizeof(Slot) * (size_t)L.P * q.S * L.M, st));
    if (ext) {
        if (xtc)
            SDTW_CUDA(launch_oimg(pr, L.P, L.N, L.M, L.D, at<char>(ws, L.ximg), at<char>(ws, L.yimg),
                                  at<char>(ws, L.xnorm), at<char>(ws, L.ynorm), st));
        if (cost) {
            SDTW_CUDA(launch_skew_cost(cost, L.P, L.N, L.M, true, at<float>(ws, L.dsk), st));
        } else if (!fused) {
            if (xtc)
                SDTW_CUDA(launch_dist_xtc(L.P, L.N, L.M, L.D, at<char>(ws, L.ximg), at<char>(ws, L.yimg),
                                          at<char>(ws, L.xnorm), at<char>(ws, L.ynorm), at<float2>(ws, L.dsk),
                                          at<int>(ws, L.status), st));
            else
                SDTW_CUDA(launch_dist_skewed_x(pr, L.P, L.N, L.M, L.D, at<float2>(ws, L.dsk), st));
        }
        q.loss = loss_out;
        q.skip_publish = debug_take_skip_publish();
        if (fused && xtc) {
            SDTW_CUDA(launch_forward_xtc(q, at<char>(ws, L.ximg), at<char>(ws, L.yimg), at<char>(ws, L.xnorm),
                                         at<char>(ws, L.ynorm), st));
        } else {
            SDTW_CUDA(launch_forward_x(q, fused, st));
        }
        return SDTW_OK;
    }
    if (tc)
        SDTW_CUDA(launch_simg(pr, L.P, L.N, L.M, L.D, at<float>(ws, L.ximg), at<float>(ws, L.yimg),
                              at<float>(ws, L.xnorm), at<float>(ws, L.ynorm), st));
    if (cost) {
        SDTW_CUDA(launch_skew_cost(cost, L.P, L.N, L.M, false, at<float>(ws, L.dsk), st));
    } else if (!fused) {
        if (tc) {
            SDTW_CUDA(launch_dist_tc(L.P, L.N, L.M, L.D, at<float>(ws, L.ximg), at<float>(ws, L.yimg),
                                     at<float>(ws, L.xnorm), at<float>(ws, L.ynorm), at<float>(ws, L.dsk),
                                     at<int>(ws, L.status), st));
        } else {
            SDTW_CUDA(launch_dist_skewed(pr, L.P, L.N, L.M, L.D, at<float>(ws, L.dsk), st));
        }
    }
    q.loss = loss_out;
    q.skip_publish = debug_take_skip_publish();
    if (L.ckpt) {  // the strips' boundary rows (edge_f), and the state of the last band, which the
                   // backward takes first: into the band buffer the backward reads it from
        const int SB = (L.NB + kBandBlocks - 1) / kBandBlocks;
        const int rb0 = (SB - 1) * kBandBlocks;
        q.VH = at<float2>(ws, L.vh) + (size_t)((SB - 1) & 1) * L.band_slots;
        q.vh_rb0 = rb0;
        q.vh_nb = L.NB - rb0 < kBandBlocks ? L.NB - rb0 : kBandBlocks;
    }
    if (fused && tc)
        SDTW_CUDA(launch_forward_tc(q, at<float>(ws, L.ximg), at<float>(ws, L.yimg), at<float>(ws, L.xnorm),
                                    at<float>(ws, L.ynorm), st));
    else
        SDTW_CUDA(launch_forward(q, fused, st));
    return SDTW_OK;
}

// Checkpointed backward with gradients: for each band of kBandBlocks row blocks, from
// the last band up, recompute the band's forward state from the boundary row the
// forward kept above it, run the band's backward wavefront (its lower boundary
// messages come from the band below, run just before), then the band's share of the
// gradient contractions: its rows of grad_x, and its rows' terms of grad_y, which
// accumulate over the bands. The state and E of two bands are kept: while band k's
// backward and gradients run on the caller's stream, band k-1 is recomputed into
// the other buffer on a side stream, once band k+1's gradients have released it.
// Every recompute runs on the side stream, so no two of them overlap (they share
// the forward's strip ticket).
sdtw_status run_backward_ckpt(const Problems& pr, const Layout& L, void* ws, float gamma, int mode,
                              const float* grad_loss, float* grad_x, float* grad_y, cudaStream_t st,
                              const int* lens_n, const int* lens_m)
{
    const int SB = (L.NB + kBandBlocks - 1) / kBandBlocks;
    int* status = at<int>(ws, L.status);
    // the band backwards on bs, the recomputes on side (both high priority: they are
    // the chain), the gradient terms on gs
    cudaStream_t bs = chain_stream(0), side = chain_stream(1), gs = grad_stream();
    cudaEvent_t ev_fork = cached_event(kEvCkptFork), ev_join = cached_event(kEvCkptJoin);
    cudaEvent_t ev_join_chain = cached_event(kEvCkptJoinChain);
    cudaEvent_t ev_rec[2] = {cached_event(kEvCkptRec0), cached_event(kEvCkptRec1)};
    cudaEvent_t ev_free[2] = {cached_event(kEvCkptFree0), cached_event(kEvCkptFree1)};
    cudaEvent_t ev_bwd[2] = {cached_event(kEvCkptBwd0), cached_event(kEvCkptBwd1)};
    if (!bs || !side || !gs || !ev_join_chain || !ev_fork || !ev_join || !ev_rec[0] || !ev_rec[1] || !ev_free[0] ||
        !ev_free[1] || !ev_bwd[0] || !ev_bwd[1])
        return SDTW_ERR_CUDA;
    WaveParams qb0 = wave_params(pr, L, ws, gamma, true, false, true);
    if (SB > 1) SDTW_CUDA(cudaMemsetAsync(qb0.edge_b, 0, 2 * sizeof(Slot) * (size_t)L.P * SB * L.M, st));
    // every band launch's counters start at zero, off the chain of band launches
    SDTW_CUDA(cudaMemsetAsync(at<char>(ws, L.ctrl_band), 0, L.ctrl_band_stride * SB, st));
    auto band_ctrl = [&](int k) { return reinterpret_cast<int*>(at<char>(ws, L.ctrl_band) + L.ctrl_band_stride * k); };
    GradParams g{};
    g.pr = pr;
    g.P = L.P; g.M = L.M; g.D = L.D;
    g.grad_loss = grad_loss;
    g.wmod = L.P;
    g.omod = L.P;
    g.coef = 1.f;
    float* img_rows = at<float>(ws, L.bimg);
    float* img_cols = at<float>(ws, L.bimg2);
    float2* vh_buf[2] = {at<float2>(ws, L.vh), at<float2>(ws, L.vh) + L.band_slots};
    float* e_buf[2] = {at<float>(ws, L.e), at<float>(ws, L.e) + L.band_slots};
    if (grad_x) {  // [Y | 1] does not depend on the band
        g.N = L.N;
        SDTW_CUDA(launch_bimg(g, img_rows, nullptr, st));
    }
    // The helper streams start after everything before this call on the caller's
    // stream, which includes the forward: it left the last band's state in buffer
    // (SB - 1) & 1, so that band needs no recompute.
    SDTW_CUDA(cudaEventRecord(ev_fork, st));
    SDTW_CUDA(cudaStreamWaitEvent(bs, ev_fork, 0));
    SDTW_CUDA(cudaStreamWaitEvent(side, ev_fork, 0));
    SDTW_CUDA(cudaStreamWaitEvent(gs, ev_fork, 0));
    SDTW_CUDA(cudaEventRecord(ev_rec[(SB - 1) & 1], st));
    // band k's forward state, recomputed from the kept boundary row above it, into buffer k % 2
    auto recompute = [&](int k, cudaStream_t s) -> sdtw_status {
        const int rb0 = k * kBandBlocks;
        const int nb = L.NB - rb0 < kBandBlocks ? L.NB - rb0 : kBandBlocks;
        WaveParams qf = wave_params(pr, L, ws, gamma, true, false, false);
        qf.W = kBandBlocks; qf.S = 1; qf.strip0 = k; qf.S_all = SB;
        qf.vh_rb0 = rb0; qf.vh_nb = nb; qf.no_loss = 1;
        qf.VH = vh_buf[k & 1];
        qf.lens_n = lens_n; qf.lens_m = lens_m;
        qf.ticket_f = band_ctrl(k);
        qf.done = band_ctrl(k) + 1;
        SDTW_CUDA(launch_forward_tc(qf, at<float>(ws, L.ximg), at<float>(ws, L.yimg), at<float>(ws, L.xnorm),
                                    at<float>(ws, L.ynorm), s));
        return SDTW_OK;
    };
    // Per band, from the last up: its backward on bs, its gradient terms on the
    // gradient stream (overlapping the next band's backward), and the next band's
    // recompute on the side stream. Buffer k % 2 holds band k's state
    // and E: the recompute of band k - 1 waits for band k + 1's backward (its state
    // buffer), band k's backward for band k + 2's gradient terms (its E buffer).
    sdtw_status s = SDTW_OK;
    for (int k = SB - 1; k >= 0 && s == SDTW_OK; --k) {
        const int rb0 = k * kBandBlocks;
        const int nb = L.NB - rb0 < kBandBlocks ? L.NB - rb0 : kBandBlocks;
        const int row0 = 32 * rb0;
        const int nrows = L.N - row0 < 32 * kBandBlocks ? L.N - row0 : 32 * kBandBlocks;
        if (k >= 1) {
            if (k + 1 < SB) SDTW_CUDA(cudaStreamWaitEvent(side, ev_bwd[(k + 1) & 1], 0));
            if ((s = recompute(k - 1, side)) != SDTW_OK) break;
            SDTW_CUDA(cudaEventRecord(ev_rec[(k - 1) & 1], side));
        }
        // the band's backward wavefront, once its state is there and its E buffer free
        SDTW_CUDA(cudaStreamWaitEvent(bs, ev_rec[k & 1], 0));
        if (k + 2 < SB) SDTW_CUDA(cudaStreamWaitEvent(bs, ev_free[k & 1], 0));
        WaveParams qb = wave_params(pr, L, ws, gamma, true, false, true);
        qb.W = kBandBlocks; qb.S = 1; qb.strip0 = k; qb.S_all = SB;
        qb.vh_rb0 = rb0; qb.vh_nb = nb;
        qb.VH = vh_buf[k & 1];
        qb.E = e_buf[k & 1];
        qb.lens_n = lens_n; qb.lens_m = lens_m;
        qb.ticket_b = band_ctrl(k) + 1 + L.P;
        SDTW_CUDA(launch_backward(qb, bs));
        SDTW_CUDA(cudaEventRecord(ev_bwd[k & 1], bs));
        // the band's gradient terms: E of the band is a problem of nrows x M. The band's
        // [X | 1] image depends on x only: it is built before waiting for the backward.
        g.E = e_buf[k & 1];
        g.pr.xs[0] = pr.xs[0] + (size_t)row0 * L.D;
        g.N = nrows;
        if (grad_y) SDTW_CUDA(launch_bimg(g, nullptr, img_cols, gs));
        SDTW_CUDA(cudaStreamWaitEvent(gs, ev_bwd[k & 1], 0));
        if (grad_x) {
            g.out = grad_x + (size_t)row0 * L.D;
            g.out_stride = (long long)L.N * L.D;
            g.accumulate = 0;
            SDTW_CUDA(launch_grad_tc(g, false, img_rows, status, gs));
        }
        if (grad_y) {
            g.out = grad_y;
            g.out_stride = (long long)L.M * L.D;
            g.accumulate = k < SB - 1;
            SDTW_CUDA(launch_grad_tc(g, true, img_cols, status, gs));
        }
        SDTW_CUDA(cudaEventRecord(ev_free[k & 1], gs));
    }
    // the helper streams' work stays ordered before anything later on the caller's
    // stream, also after an error
    cudaEventRecord(ev_join, gs);
    cudaStreamWaitEvent(st, ev_join, 0);
    cudaEventRecord(ev_join_chain, bs);
    cudaStreamWaitEvent(st, ev_join_chain, 0);
    if (s != SDTW_OK) {
        cudaEventRecord(ev_fork, side);
        cudaStreamWaitEvent(st, ev_fork, 0);
    }
    return s;
}

sdtw_status run_backward(const Problems& pr, const Layout& L, void* ws, float gamma, int mode, cudaStream_t st,
                         const int* lens_n = nullptr, const int* lens_m = nullptr)
{
    WaveParams q = wave_params(pr, L, ws, gamma, (mode & SDTW_FUSED) != 0, (mode & SDTW_EXTENDED) != 0, true);
    q.lens_n = lens_n;
    q.lens_m = lens_m;
    SDTW_CUDA(cudaMemsetAsync(at<char>(ws, L.ctrl_b), 0, L.ctrl_b_bytes, st));
    if (q.S > 1) SDTW_CUDA(cudaMemsetAsync(q.edge_b, 0, 2 * sizeof(Slot) * (size_t)L.P * q.S * L.M, st));
    SDTW_CUDA(launch_backward(q, st));
    return SDTW_OK;
}

// Gradient contractions of the problems of one set (B problems starting at set*B).
// Gradients: tensor-core GEMM form (egemm.cu) by default; the difference form
// (grad.cu, FP32 pipe) in the extended-precision mode, where rows or columns
// that align to many cells make the GEMM form cancel beyond fp32.
GradParams grad_params(const Problems& all, int set, int B, const Layout& L, void* ws)
{
    GradParams g{};
    g.pr = all;
    g.pr.xs[0] = all.xs[set]; g.pr.ys[0] = all.ys[set];
    g.pr.xstride[0] = all.xstride[set]; g.pr.ystride[0] = all.ystride[set];
    g.pr.B = B;
    g.P = B; g.N = L.N; g.M = L.M; g.D = L.D;
    g.E = at<float>(ws, L.e) + (size_t)set * B * skew_slots(L.N, L.M);
    return g;
}

// Helper streams per device for work that can overlap the caller's stream (created
// once, non-blocking; ordered against the caller's stream by events): slot 0 the
// side stream, slot 1 the checkpointed backward's gradient stream.
cudaStream_t helper_stream(int slot)
{
    static std::mutex mu;
    static cudaStream_t streams[2][64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    cudaStream_t& s = streams[slot][dev];
    if (!s && cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) s = nullptr;
    return s;
}
cudaStream_t side_stream() { return helper_stream(0); }
cudaStream_t grad_stream() { return helper_stream(1); }

// High-priority helper streams per device for the checkpointed backward's chain of
// band wavefronts (k = 0: the band backwards, 1: the band recomputes): when SMs
// free up, the block scheduler starts their CTAs before those of the gradient
// contractions queued beside them.
cudaStream_t chain_stream(int k)
{
    static std::mutex mu;
    static cudaStream_t streams[2][64] = {};
    int dev = 0;
    if (k < 0 || k > 1 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    cudaStream_t& s = streams[k][dev];
    if (!s) {
        int least = 0, greatest = 0;
        if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) greatest = 0;
        if (cudaStreamCreateWithPriority(&s, cudaStreamNonBlocking, greatest) != cudaSuccess) s = nullptr;
    }
    return s;
}

// Events that order side-stream work against the caller's stream. Each call site
// has its own slots, created once per host thread and device and reused: a slot
// is recorded and then waited on before the same thread records it again, and
// cudaStreamWaitEvent takes the record current at the time of the call. (The
// host-batch entry calls sdtw_backward inside its chunks, hence separate slots.)
cudaEvent_t cached_event(EventSlot slot)
{
    thread_local cudaEvent_t ev[64][kEvSlots] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    cudaEvent_t& e = ev[dev][slot];
    if (!e && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) e = nullptr;
    return e;
}

// Streams on which the chunks of a host-buffer call run side by side (created
// once per device, non-blocking; ordered against the caller's stream by events).
constexpr int kMaxChunks = 8;
bool chunk_streams(cudaStream_t (&out)[kMaxChunks])
{
    static std::mutex mu;
    static cudaStream_t streams[64][kMaxChunks] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lock(mu);
    for (int c = 0; c < kMaxChunks; ++c) {
        if (!streams[dev][c] && cudaStreamCreateWithFlags(&streams[dev][c], cudaStreamNonBlocking) != cudaSuccess) {
            streams[dev][c] = nullptr;
            return false;
        }
        out[c] = streams[dev][c];
    }
    return true;
}

int host_chunks(int B, int chunks)
{
    if (chunks <= 0) chunks = 2;
    if (chunks > kMaxChunks) chunks = kMaxChunks;
    return chunks < B ? chunks : B;
}

// Device workspace of sdtw_value_and_grad_host: the aggregated status word at
// offset 0, device copies of the inputs and outputs, then one forward/backward
// workspace per chunk (sized for the largest chunk).
struct HostLayout {
    size_t x, y, gx, gy, gl, loss, ws0, ws_stride, total;
    int chunks;
};

bool make_host_layout(int B, int N, int M, int D, int mode, int chunks, HostLayout* H)
{
    if (B < 1 || N < 1 || M < 1 || D < 1) return false;
    H->chunks = host_chunks(B, chunks);
    const int bmax = (B + H->chunks - 1) / H->chunks;
    Layout L;
    if (!make_layout(SDTW_OP_FWD_BWD, bmax, N, M, D, mode, &L)) return false;
    size_t o = align_up(sizeof(int));
    H->x = o; o = align_up(o + sizeof(float) * (size_t)B * N * D);
    H->y = o; o = align_up(o + sizeof(float) * (size_t)B * M * D);
    H->gx = o; o = align_up(o + sizeof(float) * (size_t)B * N * D);
    H->gy = o; o = align_up(o + sizeof(float) * (size_t)B * M * D);
    H->gl = o; o = align_up(o + sizeof(float) * (size_t)B);
    H->loss = o; o = align_up(o + sizeof(float) * (size_t)B);
    H->ws0 = o;
    H->ws_stride = align_up(L.total);
    H->total = o + (size_t)H->chunks * H->ws_stride;
    return true;
}

// status[0] = OR of the status words of the chunk workspaces.
__global__ void gather_status_kernel(int* status, const char* ws0, size_t stride, int chunks)
{
    if (threadIdx.x == 0) {
        int v = 0;
        for (int c = 0; c < chunks; ++c) v |= *reinterpret_cast<const int*>(ws0 + (size_t)c * stride);
        *status = v;
    }
}

// Workspace of sdtw_normalized_unequal: the forward/backward workspaces of the
// three batches s(x,y) (N x M), s(x,x) (N x N) and s(y,y) (M x M), in that order;
// the first one's status word (offset 0) receives the OR of all three at the end.
struct Norm3Layout {
    Layout L[3];
    size_t off[3], total;
};

bool make_norm3_layout(int B, int N, int M, int D, int mode, Norm3Layout* H)
{
    const int n[3] = {N, N, M}, m[3] = {M, N, M};
    size_t o = 0;
    for (int k = 0; k < 3; ++k) {
        if (!make_layout(SDTW_OP_FWD_BWD, B, n[k], m[k], D, mode, &H->L[k])) return false;
        H->off[k] = o;
        o = align_up(o + H->L[k].total);
    }
    H->total = o;
    return true;
}

__global__ void gather3_status_kernel(int* out, const int* s1, const int* s2)
{
    if (threadIdx.x == 0) *out = *out | *s1 | *s2;
}

__global__ void combine3_normalized_kernel(const float* lxy, const float* lxx, const float* lyy, int B, float* loss)
{
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) loss[b] = lxy[b] - 0.5f * (lxx[b] + lyy[b]);
}

// images_ready: when not null, the operand images were already launched on
// another stream; the contractions wait on this event instead of building them.
sdtw_status run_grads(const Problems& all, int set, int B, const Layout& L, void* ws, const float* grad_loss,
                      float coef, float* out_x, float* out_y, int accumulate, int mode, cudaStream_t st,
                      cudaEvent_t images_ready = nullptr)
{
    GradParams g = grad_params(all, set, B, L, ws);
    g.grad_loss = grad_loss;
    g.wmod = B;
    g.coef = coef;
    g.omod = B;
    g.accumulate = accumulate;
    const bool simt = (mode & SDTW_EXTENDED) != 0;
    int* status = at<int>(ws, L.status);
    float* img_rows = at<float>(ws, L.bimg);
    float* img_cols = at<float>(ws, L.bimg2);
    if (!simt && images_ready) SDTW_CUDA(cudaStreamWaitEvent(st, images_ready, 0));
    else if (!simt) SDTW_CUDA(launch_bimg(g, out_x ? img_rows : nullptr, out_y ? img_cols : nullptr, st));
    if (simt) {   // the difference-form contractions visit only the tiles where E is non-zero
        int2* bounds = at<int2>(ws, L.ebnd) + (size_t)set * B * L.NB;
        SDTW_CUDA(launch_ebounds(g, bounds, st));
        g.bounds = bounds;
    }
    if (out_x) {
        g.out = out_x;
        g.out_stride = (long long)L.N * L.D;
        SDTW_CUDA(simt ? launch_grad_rows(g, st) : launch_grad_tc(g, false, img_rows, status, st));
    }
    if (out_y) {
        g.out = out_y;
        g.out_stride = (long long)L.M * L.D;
        SDTW_CUDA(simt ? launch_grad_cols(g, st) : launch_grad_tc(g, true, img_cols, status, st));
    }
    return SDTW_OK;
}

// out[i] = exp2_neg(x[i]): the library's own exp2 of the double-float path, for its test.
__global__ void exp2_neg_kernel(const float* x, float* out, int n)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) out[i] = exp2_neg(x[i]);
}

__global__ void combine_normalized_kernel(const float* l, int B, float* loss)
{
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) loss[b] = l[b] - 0.5f * (l[B + b] + l[2 * B + b]);
}

sdtw_status check_cost(const float* C, int B, int N, int M, float gamma, int mode)
{
    if (B < 1 || N < 1 || M < 1) return SDTW_ERR_EMPTY;
    if (!(gamma > 0.f) || !std::isfinite(gamma)) return SDTW_ERR_GAMMA;
    if ((mode & ~3) || (mode & SDTW_FUSED)) return SDTW_ERR_ARG;
    if (!C) return SDTW_ERR_ARG;
    if (B > 65535 / 3 || N > (1 << 24) || M > (1 << 24)) return SDTW_ERR_TOO_LARGE;
    return SDTW_OK;
}

}  // namespace

namespace sdtw {
unsigned long long debug_wait_ns() { return g_wait_ns; }
int debug_take_skip_publish()
{
    const int v = g_skip_publish;
    g_skip_publish = 0;
    return v;
}
}  // namespace sdtw

extern "C" {

size_t sdtw_workspace_bytes(int op, int B, int N, int M, int D, sdtw_mode mode)
{
    if (op == SDTW_OP_NORMALIZED_UNEQUAL) {
        Norm3Layout H;
        return make_norm3_layout(B, N, M, D, (int)mode, &H) ? H.total : 0;
    }
    Layout L;
    if (!make_layout(op, B, N, M, D, (int)mode, &L)) return 0;
    return L.total;
}

sdtw_status sdtw_distance(const float* x, const float* y, int B, int N, int M, int D, float* C, void* stream)
{
    sdtw_status s = check_common(x, y, B, N, M, D, 1.f, SDTW_UNFUSED);
    if (s != SDTW_OK) return s;
    if (!C) return SDTW_ERR_ARG;
    Problems pr{};
    pr.xs[0] = x; pr.ys[0] = y;
    pr.xstride[0] = (long long)N * D; pr.ystride[0] = (long long)M * D;
    pr.B = B;
    SDTW_CUDA(launch_dist_rowmajor(pr, B, N, M, D, C, static_cast<cudaStream_t>(stream)));
    return SDTW_OK;
}

sdtw_status sdtw_forward(const float* x, const float* y, int B, int N, int M, int D, float gamma, sdtw_mode mode,
                         float* loss, void* ws, size_t ws_bytes, void* stream)
{
    return sdtw_forward_varlen(x, y, nullptr, nullptr, B, N, M, D, gamma, mode, loss, ws, ws_bytes, stream);
}

sdtw_status sdtw_forward_varlen(const float* x, const float* y, const int* x_lengths, const int* y_lengths, int B,
                                int N, int M, int D, float gamma, sdtw_mode mode, float* loss, void* ws,
                                size_t ws_bytes, void* stream)
{
    sdtw_status s = check_common(x, y, B, N, M, D, gamma, (int)mode, true);
    if (s != SDTW_OK) return s;
    if (!loss) return SDTW_ERR_ARG;
    Layout L;
    make_layout(SDTW_OP_FWD_BWD, B, N, M, D, (int)mode, &L);
    if ((s = check_ws(ws, ws_bytes, L)) != SDTW_OK) return s;
    Problems pr{};
    pr.xs[0] = x; pr.ys[0] = y;
    pr.xstride[0] = (long long)N * D; pr.ystride[0] = (long long)M * D;
    pr.B = B;
    return run_forward(pr, L, ws, gamma, (int)mode, loss, static_cast<cudaStream_t>(stream), nullptr, x_lengths,
                       y_lengths);
}

sdtw_status sdtw_backward(const float* x, const float* y, int B, int N, int M, int D, float gamma, sdtw_mode mode,
                          const float* grad_loss, float* grad_x, float* grad_y, void* ws, size_t ws_bytes,
                          void* stream)
{
    return sdtw_backward_varlen(x, y, nullptr, nullptr, B, N, M, D, gamma, mode, grad_loss, grad_x, grad_y, ws,
                                ws_bytes, stream);
}

sdtw_status sdtw_backward_varlen(const float* x, const float* y, const int* x_lengths, const int* y_lengths, int B,
                                 int N, int M, int D, float gamma, sdtw_mode mode, const float* grad_loss,
                                 float* grad_x, float* grad_y, void* ws, size_t ws_bytes, void* stream)
{
    sdtw_status s = check_common(x, y, B, N, M, D, gamma, (int)mode, true);
    if (s != SDTW_OK) return s;
    if (!grad_loss) return SDTW_ERR_ARG;
    Layout L;
    make_layout(SDTW_OP_FWD_BWD, B, N, M, D, (int)mode, &L);
    if ((s = check_ws(ws, ws_bytes, L)) != SDTW_OK) return s;
    Problems pr{};
    pr.xs[0] = x; pr.ys[0] = y;
    pr.xstride[0] = (long long)N * D; pr.ystride[0] = (long long)M * D;
    pr.B = B;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (L.ckpt) {
        return run_backward_ckpt(pr, L, ws, gamma, (int)mode, grad_loss, grad_x, grad_y, st, x_lengths, y_lengths);
    }
    // The gradient operand images depend on x and y only: they are built on a side
    // stream while the backward wavefront runs (it leaves most of each SM idle).
    cudaStream_t side = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    const bool tc_grads = (grad_x || grad_y) && !(mode & SDTW_EXTENDED);
    if (tc_grads && (side = side_stream()) != nullptr && (fork = cached_event(kEvBwdFork)) != nullptr &&
        (join = cached_event(kEvBwdJoin)) != nullptr) {
        GradParams g = grad_params(pr, 0, B, L, ws);
        bool launched = cudaEventRecord(fork, st) == cudaSuccess && cudaStreamWaitEvent(side, fork, 0) == cudaSuccess &&
                        launch_bimg(g, grad_x ? at<float>(ws, L.bimg) : nullptr,
                                    grad_y ? at<float>(ws, L.bimg2) : nullptr, side) == cudaSuccess &&
                        cudaEventRecord(join, side) == cudaSuccess;
        if (!launched) return SDTW_ERR_CUDA;
    } else {
        join = nullptr;
    }
    s = run_backward(pr, L, ws, gamma, (int)mode, st, x_lengths, y_lengths);
    if (s == SDTW_OK && (grad_x || grad_y))
        s = run_grads(pr, 0, B, L, ws, grad_loss, 1.f, grad_x, grad_y, 0, (int)mode, st, join);
    if (join && s != SDTW_OK) cudaStreamWaitEvent(st, join, 0);  // keep the side work ordered before later calls
    return s;
}

}  // extern "C"

namespace {

// Normalized Soft-DTW of equal lengths over one batch of 3B problems. fwd: the
// forward and the combined losses; bwd: the backward wavefronts and the ordered
// gradient launches, reading the state the forward left in `ws`.
sdtw_status normalized_impl(const float* x, const float* y, int B, int N, int D, float gamma, int mode, float* loss,
                            const float* grad_loss, float* grad_x, float* grad_y, void* ws, size_t ws_bytes,
                            cudaStream_t st, bool fwd, bool bwd)
{
    sdtw_status s = check_common(x, y, B, N, N, D, gamma, mode);
    if (s != SDTW_OK) return s;
    if (fwd && !loss) return SDTW_ERR_ARG;
    if (!fwd && !grad_loss) return SDTW_ERR_ARG;
    Layout L;
    make_layout(SDTW_OP_NORMALIZED, B, N, N, D, mode, &L);
    if ((s = check_ws(ws, ws_bytes, L)) != SDTW_OK) return s;
    const long long st_ = (long long)N * D;
    Problems pr{};
    pr.xs[0] = x; pr.ys[0] = y;   // s(x, y)
    pr.xs[1] = x; pr.ys[1] = x;   // s(x, x)
    pr.xs[2] = y; pr.ys[2] = y;   // s(y, y)
    for (int k = 0; k < 3; ++k) { pr.xstride[k] = st_; pr.ystride[k] = st_; }
    pr.B = B;
    if (fwd) {
        float* l3 = at<float>(ws, L.losses);
        if ((s = run_forward(pr, L, ws, gamma, mode, l3, st)) != SDTW_OK) return s;
        combine_normalized_kernel<<<(B + 255) / 256, 256, 0, st>>>(l3, B, loss);
        SDTW_CUDA(cudaGetLastError());
    }
    if (!bwd || !grad_loss || (!grad_x && !grad_y)) return SDTW_OK;
    if ((s = run_backward(pr, L, ws, gamma, mode, st)) != SDTW_OK) return s;
    // grad_x = g [gx(x,y) - (gx(x,x) + gy(x,x))/2];  grad_y = g [gy(x,y) - (gx(y,y) + gy(y,y))/2]
    if ((s = run_grads(pr, 0, B, L, ws, grad_loss, 1.f, grad_x, grad_y, 0, mode, st)) != SDTW_OK) return s;
    if (grad_x) {
        if ((s = run_grads(pr, 1, B, L, ws, grad_loss, -0.5f, grad_x, grad_x, 1, mode, st)) != SDTW_OK) return s;
    }
    if (grad_y) {
        if ((s = run_grads(pr, 2, B, L, ws, grad_loss, -0.5f, grad_y, grad_y, 1, mode, st)) != SDTW_OK) return s;
    }
    return SDTW_OK;
}

// Normalized Soft-DTW of unequal lengths: three batches (N x M, N x N, M x M) on
// three streams. fwd / bwd as for normalized_impl.
sdtw_status normalized_unequal_impl(const float* x, const float* y, int B, int N, int M, int D, float gamma, int mode,
                                    float* loss, const float* grad_loss, float* grad_x, float* grad_y, void* ws,
                                    size_t ws_bytes, cudaStream_t st, bool fwd, bool bwd)
{
    sdtw_status s = check_common(x, y, B, N, M, D, gamma, mode);
    if (s != SDTW_OK) return s;
    if (fwd && !loss) return SDTW_ERR_ARG;
    if (!fwd && !grad_loss) return SDTW_ERR_ARG;
    Norm3Layout H;
    if (!make_norm3_layout(B, N, M, D, mode, &H)) return SDTW_ERR_ARG;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0 || ws_bytes < H.total) return SDTW_ERR_WORKSPACE;
    const bool grads = bwd && grad_loss && (grad_x || grad_y);
    if (!fwd && !grads) return SDTW_OK;
    Problems pr[3] = {};
    const float* xs[3] = {x, x, y};
    const float* ys[3] = {y, x, y};
    const long long xst[3] = {(long long)N * D, (long long)N * D, (long long)M * D};
    const long long yst[3] = {(long long)M * D, (long long)N * D, (long long)M * D};
    void* wsk[3];
    for (int k = 0; k < 3; ++k) {
        pr[k].xs[0] = xs[k]; pr[k].ys[0] = ys[k];
        pr[k].xstride[0] = xst[k]; pr[k].ystride[0] = yst[k];
        pr[k].B = B;
        wsk[k] = at<char>(ws, H.off[k]);
    }
    cudaStream_t cs[kMaxChunks];
    if (!chunk_streams(cs)) return SDTW_ERR_CUDA;
    // The three wavefront pairs are independent and latency-bound: they run side by
    // side on three streams, each sized for a third of the SMs.
    cudaEvent_t fork = cached_event(kEvNormFork), join = cached_event(kEvNormJoin);
    if (!fork || !join || cudaEventRecord(fork, st) != cudaSuccess) return SDTW_ERR_CUDA;
    const int prev_share = t_sm_share;
    t_sm_share = num_sms() / 3 > 0 ? num_sms() / 3 : 1;
    for (int k = 0; k < 3; ++k) {
        if (s == SDTW_OK && cudaStreamWaitEvent(cs[k], fork, 0) != cudaSuccess) s = SDTW_ERR_CUDA;
        if (s == SDTW_OK && fwd)
            s = run_forward(pr[k], H.L[k], wsk[k], gamma, mode, at<float>(wsk[k], H.L[k].losses), cs[k]);
        if (s == SDTW_OK && grads) s = run_backward(pr[k], H.L[k], wsk[k], gamma, mode, cs[k]);
        // joined whatever happened, so later work stays ordered
        if ((cudaEventRecord(join, cs[k]) != cudaSuccess || cudaStreamWaitEvent(st, join, 0) != cudaSuccess) &&
            s == SDTW_OK)
            s = SDTW_ERR_CUDA;
    }
    t_sm_share = prev_share;
    if (s != SDTW_OK) return s;
    if (fwd) {
        combine3_normalized_kernel<<<(B + 255) / 256, 256, 0, st>>>(at<float>(wsk[0], H.L[0].losses),
                                                                    at<float>(wsk[1], H.L[1].losses),
                                                                    at<float>(wsk[2], H.L[2].losses), B, loss);
        SDTW_CUDA(cudaGetLastError());
    }
    if (grads) {
        // grad_x = g [gx(x,y) - (gx(x,x) + gy(x,x))/2];  grad_y = g [gy(x,y) - (gx(y,y) + gy(y,y))/2]
        s = run_grads(pr[0], 0, B, H.L[0], wsk[0], grad_loss, 1.f, grad_x, grad_y, 0, mode, st);
        if (s == SDTW_OK && grad_x)
            s = run_grads(pr[1], 0, B, H.L[1], wsk[1], grad_loss, -0.5f, grad_x, grad_x, 1, mode, st);
        if (s == SDTW_OK && grad_y)
            s = run_grads(pr[2], 0, B, H.L[2], wsk[2], grad_loss, -0.5f, grad_y, grad_y, 1, mode, st);
        if (s != SDTW_OK) return s;
    }
    gather3_status_kernel<<<1, 32, 0, st>>>(at<int>(wsk[0], H.L[0].status), at<int>(wsk[1], H.L[1].status),
                                            at<int>(wsk[2], H.L[2].status));
    SDTW_CUDA(cudaGetLastError());
    return SDTW_OK;
}

}  // namespace

extern "C" {

sdtw_status sdtw_normalized(const float* x, const float* y, int B, int N, int D, float gamma, sdtw_mode mode,
                            float* loss, const float* grad_loss, float* grad_x, float* grad_y, void* ws,
                            size_t ws_bytes, void* stream)
{
    return normalized_impl(x, y, B, N, D, gamma, (int)mode, loss, grad_loss, grad_x, grad_y, ws, ws_bytes,
                           static_cast<cudaStream_t>(stream), true, true);
}

sdtw_status sdtw_normalized_backward(const float* x, const float* y, int B, int N, int D, float gamma,
                                     sdtw_mode mode, const float* grad_loss, float* grad_x, float* grad_y, void* ws,
                                     size_t ws_bytes, void* stream)
{
    return normalized_impl(x, y, B, N, D, gamma, (int)mode, nullptr, grad_loss, grad_x, grad_y, ws, ws_bytes,
                           static_cast<cudaStream_t>(stream), false, true);
}

sdtw_status sdtw_barycenter_step(float* z, float* m, float* v, int t, const float* X, int K, int T, int T2, int D,
                                 float gamma, float lr, float beta1, float beta2, float eps, sdtw_mode mode,
                                 float* loss_out, void* ws, size_t ws_bytes, void* stream)
{
    return sdtw_barycenter_step_clipped(z, m, v, t, X, K, T, T2, D, gamma, lr, beta1, beta2, eps, 0.f, mode,
                                        loss_out, ws, ws_bytes, stream);
}

sdtw_status sdtw_barycenter_step_clipped(float* z, float* m, float* v, int t, const float* X, int K, int T, int T2,
                                         int D, float gamma, float lr, float beta1, float beta2, float eps,
                                         float max_grad_norm, sdtw_mode mode, float* loss_out, void* ws,
                                         size_t ws_bytes, void* stream)
{
    sdtw_status s = check_common(z, X, K, T, T2, D, gamma, (int)mode);
    if (s != SDTW_OK) return s;
    if (!m || !v || t < 1 || !(lr >= 0.f) || !(beta1 >= 0.f && beta1 < 1.f) || !(beta2 >= 0.f && beta2 < 1.f) ||
        !(eps >= 0.f) || !(max_grad_norm >= 0.f))
        return SDTW_ERR_ARG;
    Layout L;
    make_layout(SDTW_OP_BARYCENTER, K, T, T2, D, (int)mode, &L);
    if ((s = check_ws(ws, ws_bytes, L)) != SDTW_OK) return s;
    Problems pr{};
    pr.xs[0] = z; pr.ys[0] = X;
    pr.xstride[0] = 0;                      // z broadcast against every sequence
    pr.ystride[0] = (long long)T2 * D;
    pr.B = K;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float* losses = at<float>(ws, L.losses);
    if ((s = run_forward(pr, L, ws, gamma, (int)mode, losses, st)) != SDTW_OK) return s;
    if ((s = run_backward(pr, L, ws, gamma, (int)mode, st)) != SDTW_OK) return s;
    float* gparts = at<float>(ws, L.gparts);
    if ((s = run_grads(pr, 0, K, L, ws, nullptr, 1.f / (float)K, gparts, nullptr, 0, (int)mode, st)) != SDTW_OK)
        return s;
    const double bc1 = 1.0 - std::pow((double)beta1, (double)t);
    const double bc2 = 1.0 - std::pow((double)beta2, (double)t);
    if (max_grad_norm > 0.f)
        SDTW_CUDA(launch_adam_clipped(z, m, v, gparts, K, T * D, lr, beta1, beta2, eps, (float)bc1, (float)bc2,
                                      max_grad_norm, at<float>(ws, L.gnorm), losses, loss_out, st));
    else
        SDTW_CUDA(launch_adam(z, m, v, gparts, K, T * D, lr, beta1, beta2, eps, (float)bc1, (float)bc2, losses,
                              loss_out, st));
    return SDTW_OK;
}

sdtw_status sdtw_forward_cost(const float* C, int B, int N, int M, float gamma, sdtw_mode mode, float* loss,
                              void* ws, size_t ws_bytes, void* stream)
{
    sdtw_status s = check_cost(C, B, N, M, gamma, (int)mode);
    if (s != SDTW_OK) return s;
    if (!loss) return SDTW_ERR_ARG;
    Layout L;
    make_layout(SDTW_OP_COST, B, N, M, 1, (int)mode, &L);
    if ((s = check_ws(ws, ws_bytes, L)) != SDTW_OK) return s;
    Problems pr{};
    pr.B = B;
    return run_forward(pr, L, ws, gamma, (int)mode, loss, static_cast<cudaStream_t>(stream), C);
}

sdtw_status sdtw_backward_cost(const float* C, int B, int N, int M, float gamma, sdtw_mode mode,
                               const float* grad_loss, float* grad_C, void* ws, size_t ws_bytes, void* stream)
{
    sdtw_status s = check_cost(C, B, N, M, gamma, (int)mode);
    if (s != SDTW_OK) return s;
    if (!grad_loss || !grad_C) return SDTW_ERR_ARG;
    Layout L;
    make_layout(SDTW_OP_COST, B, N, M, 1, (int)mode, &L);
    if ((s = check_ws(ws, ws_bytes, L)) != SDTW_OK) return s;
    Problems pr{};
    pr.B = B;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if ((s = run_backward(pr, L, ws, gamma, (int)mode, st)) != SDTW_OK) return s;
    SDTW_CUDA(launch_unskew_grad(at<float>(ws, L.e), B, N, M, grad_loss, grad_C, st));
    return SDTW_OK;
}

sdtw_status sdtw_normalized_unequal(const float* x, const float* y, int B, int N, int M, int D, float gamma,
                                    sdtw_mode mode, float* loss, const float* grad_loss, float* grad_x,
                                    float* grad_y, void* ws, size_t ws_bytes, void* stream)
{
    return normalized_unequal_impl(x, y, B, N, M, D, gamma, (int)mode, loss, grad_loss, grad_x, grad_y, ws, ws_bytes,
                                   static_cast<cudaStream_t>(stream), true, true);
}

sdtw_status sdtw_normalized_unequal_backward(const float* x, const float* y, int B, int N, int M, int D,
                                             float gamma, sdtw_mode mode, const float* grad_loss, float* grad_x,
                                             float* grad_y, void* ws, size_t ws_bytes, void* stream)
{
    return normalized_unequal_impl(x, y, B, N, M, D, gamma, (int)mode, nullptr, grad_loss, grad_x, grad_y, ws,
                                   ws_bytes, static_cast<cudaStream_t>(stream), false, true);
}

size_t sdtw_host_workspace_bytes(int B, int N, int M, int D, sdtw_mode mode, int chunks)
{
    HostLayout H;
    if (!make_host_layout(B, N, M, D, (int)mode, chunks, &H)) return 0;
    return H.total;
}

sdtw_status sdtw_value_and_grad_host(const float* x, const float* y, const float* grad_loss, int B, int N, int M,
                                     int D, float gamma, sdtw_mode mode, float* loss, float* grad_x, float* grad_y,
                                     int chunks, void* ws, size_t ws_bytes, void* stream)
{
    sdtw_status s = check_common(x, y, B, N, M, D, gamma, (int)mode);
    if (s != SDTW_OK) return s;
    const bool grads = grad_x || grad_y;
    if (!loss || (grads && !grad_loss)) return SDTW_ERR_ARG;
    HostLayout H;
    if (!make_host_layout(B, N, M, D, (int)mode, chunks, &H)) return SDTW_ERR_ARG;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0 || ws_bytes < H.total) return SDTW_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaStream_t cs[kMaxChunks];
    if (!chunk_streams(cs)) return SDTW_ERR_CUDA;
    cudaEvent_t fork = cached_event(kEvHostFork), join = cached_event(kEvHostJoin);
    if (!fork || !join || cudaEventRecord(fork, st) != cudaSuccess) return SDTW_ERR_CUDA;
    const int prev_share = t_sm_share;
    t_sm_share = num_sms() / H.chunks > 0 ? num_sms() / H.chunks : 1;
    const size_t xr = (size_t)N * D, yr = (size_t)M * D;  // floats per problem
    const auto h2d = cudaMemcpyHostToDevice;
    const auto d2h = cudaMemcpyDeviceToHost;
    for (int c = 0; c < H.chunks && s == SDTW_OK; ++c) {
        const int b0 = (int)((long long)c * B / H.chunks), b1 = (int)((long long)(c + 1) * B / H.chunks);
        const int Bc = b1 - b0;
        cudaStream_t sc = cs[c];
        float* xd = at<float>(ws, H.x) + b0 * xr;
        float* yd = at<float>(ws, H.y) + b0 * yr;
        float* gxd = grad_x ? at<float>(ws, H.gx) + b0 * xr : nullptr;
        float* gyd = grad_y ? at<float>(ws, H.gy) + b0 * yr : nullptr;
        float* gld = at<float>(ws, H.gl) + b0;
        float* lossd = at<float>(ws, H.loss) + b0;
        void* wsc = at<char>(ws, H.ws0 + (size_t)c * H.ws_stride);
        // inputs of this chunk in, its forward and backward, its outputs out: the copies
        // of one chunk overlap the kernels of the others
        bool ok = cudaStreamWaitEvent(sc, fork, 0) == cudaSuccess &&
                  cudaMemcpyAsync(xd, x + b0 * xr, sizeof(float) * Bc * xr, h2d, sc) == cudaSuccess &&
                  cudaMemcpyAsync(yd, y + b0 * yr, sizeof(float) * Bc * yr, h2d, sc) == cudaSuccess &&
                  (!grads || cudaMemcpyAsync(gld, grad_loss + b0, sizeof(float) * Bc, h2d, sc) == cudaSuccess);
        if (!ok) s = SDTW_ERR_CUDA;
        if (s == SDTW_OK) s = sdtw_forward(xd, yd, Bc, N, M, D, gamma, mode, lossd, wsc, H.ws_stride, sc);
        if (s == SDTW_OK && grads)
            s = sdtw_backward(xd, yd, Bc, N, M, D, gamma, mode, gld, gxd, gyd, wsc, H.ws_stride, sc);
        if (s == SDTW_OK) {
            ok = cudaMemcpyAsync(loss + b0, lossd, sizeof(float) * Bc, d2h, sc) == cudaSuccess &&
                 (!grad_x || cudaMemcpyAsync(grad_x + b0 * xr, gxd, sizeof(float) * Bc * xr, d2h, sc) == cudaSuccess) &&
                 (!grad_y || cudaMemcpyAsync(grad_y + b0 * yr, gyd, sizeof(float) * Bc * yr, d2h, sc) == cudaSuccess);
            if (!ok) s = SDTW_ERR_CUDA;
        }
        // join, whatever happened, so that later work on the caller's stream stays ordered
        if ((cudaEventRecord(join, sc) != cudaSuccess || cudaStreamWaitEvent(st, join, 0) != cudaSuccess) &&
            s == SDTW_OK)
            s = SDTW_ERR_CUDA;
    }
    t_sm_share = prev_share;
    if (s != SDTW_OK) return s;
    gather_status_kernel<<<1, 32, 0, st>>>(at<int>(ws, 0), at<char>(ws, H.ws0), H.ws_stride, H.chunks);
    SDTW_CUDA(cudaGetLastError());
    return SDTW_OK;
}

sdtw_status sdtw_last_device_status(void* ws, void* stream)
{
    if (!ws) return SDTW_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return SDTW_ERR_CUDA;
    int h = 0;
    if (cudaMemcpy(&h, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SDTW_ERR_CUDA;
    if (h == 0) return SDTW_OK;
    if (cudaMemset(ws, 0, sizeof(int)) != cudaSuccess) return SDTW_ERR_CUDA;
    return SDTW_ERR_TIMEOUT;
}

const char* sdtw_status_string(sdtw_status s)
{
    switch (s) {
        case SDTW_OK: return "ok";
        case SDTW_ERR_ARG: return "invalid argument";
        case SDTW_ERR_GAMMA: return "gamma must be finite and > 0";
        case SDTW_ERR_EMPTY: return "empty input (B, N, M and D must be >= 1)";
        case SDTW_ERR_SHAPE: return "shape mismatch";
        case SDTW_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case SDTW_ERR_CUDA: return "CUDA runtime or launch error";
        case SDTW_ERR_TIMEOUT: return "device-side wait timed out";
        case SDTW_ERR_TOO_LARGE: return "sizes exceed the library's limits";
    }
    return "unknown status";
}

void sdtw_debug_set_wait(double seconds, int skip_publish)
{
    g_wait_ns = (seconds > 0.0) ? (unsigned long long)(seconds * 1e9) : kDefaultWaitNs;
    g_skip_publish = skip_publish ? 1 : 0;
}

sdtw_status sdtw_debug_exp2_neg(const float* x, float* out, int n, void* stream)
{
    if (n < 0 || (n > 0 && (!x || !out))) return SDTW_ERR_ARG;
    if (n == 0) return SDTW_OK;
    exp2_neg_kernel<<<(n + 255) / 256, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, out, n);
    SDTW_CUDA(cudaGetLastError());
    return SDTW_OK;
}

void sdtw_debug_set_options(int warps_fwd, int warps_bwd, int dist_simt, int fused_simt)
{
    g_dbg.warps_fwd = warps_fwd > 0 ? warps_fwd : 0;
    g_dbg.warps_bwd = warps_bwd > 0 ? warps_bwd : 0;
    g_dbg.dist_simt = dist_simt ? 1 : 0;
    g_dbg.fused_simt = fused_simt ? 1 : 0;
}

void sdtw_debug_set_clusters(int max_cluster)
{
    g_dbg.max_cluster = max_cluster > 0 ? (max_cluster >= 4 ? 4 : max_cluster) : 0;
}

}  // extern "C"
