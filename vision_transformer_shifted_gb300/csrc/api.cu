// C ABI of libswin_wattn: argument checks, path choice, workspace, launches.
#include <cstdlib>
#include <cstring>
#include <new>

#include "swin_wattn.h"
#include "swin_wattn_backward.h"
#include "swin_wattn_test.h"
#include "common.cuh"

using namespace swin;

// Chunks of whole images of the pipelined host-buffer forward (at most).
constexpr int HOST_CHUNKS = 16;   // most chunks of the host-buffer forward (default 8)

struct swin_wattn_s {
    int C, heads, d, M, shift, mode;
    bool fp32;
    int path_opt;
    uint64_t wait_ns;
    int device;
    int *d_err;
    void *ws;          // three-kernel workspace: qkv [T,3C] then attn [T,C] (bf16)
    size_t ws_bytes;
    void *stage_x, *stage_out; // device staging of swin_wattn_forward_host
    size_t stage_bytes;
    int last_launches;
    cudaError_t last_cuda_error;
    void *bws;         // backward workspace (see swin_wattn_backward)
    size_t bws_bytes;
    int bw_launches;
    // chunked host-buffer forward: copy-in, compute and copy-out streams and
    // their events (created on first use)
    cudaStream_t hs[3];
    cudaEvent_t ev_in[HOST_CHUNKS], ev_run[HOST_CHUNKS], ev_fork, ev_join, ev_done;
    bool hs_ready;
    // the chunked pipeline captured as a CUDA graph, replayed while the call's
    // arguments stay the same
    cudaGraphExec_t graph;
    const void *g_args[11];   // the call's pointers and the buffers the graph uses
    int g_B, g_H, g_W, g_path, g_launches, g_chunks;
    int host_chunks;   // chunks of the host-buffer forward (1..HOST_CHUNKS)
    int overlap;       // SWIN_WATTN_OPT_OVERLAP_CALLS
};

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? SWIN_WATTN_OK : SWIN_WATTN_ECUDA; }

size_t elem_bytes(const swin_wattn_s *h) { return h->fp32 ? 4 : 2; }

// Shape checks shared by every entry point that takes B, H, W.
int check_grid(const swin_wattn_s *h, int B, int H, int W)
{
    if (B < 0 || H <= 0 || W <= 0) return SWIN_WATTN_EINVAL;
    if (H % h->M || W % h->M) return SWIN_WATTN_EINVAL;
    if ((int64_t)B * H * W * h->C > (int64_t)1 << 40) return SWIN_WATTN_EINVAL;
    return SWIN_WATTN_OK;
}

// The fused kernel indexes tokens with 32-bit integers: grids of 2^31 tokens
// or more take the three-kernel path.
int choose_path(const swin_wattn_s *h, int64_t T)
{
    if (h->fp32) return 3;
    return fused_supported(h->M, h->C, h->heads) && T < ((int64_t)1 << 31) ? 2 : 1;
}

DeviceStatus dstatus(const swin_wattn_s *h) { return DeviceStatus{h->d_err, h->wait_ns}; }

// Guard bands (SWIN_WATTN_DEBUG) of the buffers the host-buffer forward uses.
int check_host_guards(const swin_wattn_s *h, cudaStream_t s)
{
    for (const void *b : {h->stage_x, h->stage_out, h->ws}) {
        const int rc = ws_check(b, s);
        if (rc) return rc;
    }
    return SWIN_WATTN_OK;
}

// (overlap: the fused kernel may start while the stream's earlier kernels
// finish, see SWIN_WATTN_OPT_OVERLAP_CALLS)
int run_forward(swin_wattn_s *h, const void *x, int B, int H, int W, const void *Wqkv, const void *bqkv,
                const void *table, const float *tau, const void *Wproj, const void *bproj, void *out,
                cudaStream_t stream, bool overlap = false)
{
    const Geom g = make_geom(B, H, W, h->C, h->M, h->shift);
    h->last_launches = 0;
    if (B == 0) return SWIN_WATTN_OK;
    const int path = h->path_opt ? h->path_opt : choose_path(h, g.T);
    if (h->fp32) {
        Fp32Args a;
        a.x = (const float *)x; a.Wqkv = (const float *)Wqkv; a.bqkv = (const float *)bqkv;
        a.table = (const float *)table; a.tau = tau; a.Wproj = (const float *)Wproj; a.bproj = (const float *)bproj;
        a.out = (float *)out; a.heads = h->heads; a.mode = h->mode; a.g = g;
        cudaError_t e = launch_fp32_block(a, stream);
        if (e == cudaErrorInvalidConfiguration) return SWIN_WATTN_EUNSUPPORTED;
        if (e != cudaSuccess) h->last_cuda_error = e;
        h->last_launches = 1;
        return cuda_status(e);
    }
    if (path == 2) {
        if (!fused_supported(h->M, h->C, h->heads) || g.T >= ((int64_t)1 << 31)) return SWIN_WATTN_EUNSUPPORTED;
        cudaError_t e = launch_fused((const bf16 *)x, (const bf16 *)Wqkv, (const bf16 *)bqkv, (const bf16 *)table, tau,
                                     (const bf16 *)Wproj, (const bf16 *)bproj, (bf16 *)out, h->mode, g, dstatus(h),
                                     h->d_err + 2, stream, nullptr, nullptr, 0, overlap ? 1 : 0);
        if (e != cudaSuccess) {
            h->last_cuda_error = e;
            return SWIN_WATTN_ECUDA;
        }
        h->last_launches = 1;
        return SWIN_WATTN_OK;
    }
    if (path != 1) return SWIN_WATTN_EUNSUPPORTED;
    const size_t qkv_bytes = (size_t)g.T * 3 * h->C * 2, attn_bytes = (size_t)g.T * h->C * 2;
    int rc = ws_ensure(&h->ws, &h->ws_bytes, qkv_bytes + attn_bytes);
    if (rc) return rc;
    bf16 *qkv = (bf16 *)h->ws;
    bf16 *attn = (bf16 *)((char *)h->ws + qkv_bytes);
    GemmArgs k1{};
    k1.A = (const bf16 *)x; k1.lda = h->C; k1.Bw = (const bf16 *)Wqkv; k1.bias = (const bf16 *)bqkv;
    k1.D = qkv; k1.ldd = 3 * h->C; k1.rows = g.T; k1.N = 3 * h->C; k1.K = h->C; k1.g = g;
    k1.norm_cols = h->mode == SWIN_WATTN_V2 ? 2 * h->C : 0;
    // (overlap: each kernel's prologue -- weights, tables -- runs while the one
    // before it finishes; the workspace is written only after the previous
    // kernel, and so every earlier one, has completed)
    k1.overlap = overlap ? 1 : 0;
    cudaError_t e = launch_gemm(k1, LOAD_GATHER, STORE_PLAIN, dstatus(h), stream);
    if (e != cudaSuccess) { h->last_cuda_error = e; return SWIN_WATTN_ECUDA; }
    AttnArgs k2{};
    k2.qkv = qkv; k2.attn = attn; k2.table = (const bf16 *)table; k2.tau = tau; k2.heads = h->heads;
    k2.mode = h->mode; k2.g = g; k2.overlap = overlap ? 1 : 0;
    e = launch_attention(k2, dstatus(h), stream);
    if (e != cudaSuccess) { h->last_cuda_error = e; return SWIN_WATTN_ECUDA; }
    GemmArgs k3{};
    k3.A = attn; k3.lda = h->C; k3.Bw = (const bf16 *)Wproj; k3.bias = (const bf16 *)bproj;
    k3.D = (bf16 *)out; k3.ldd = h->C; k3.rows = g.T; k3.N = h->C; k3.K = h->C; k3.g = g;
    k3.overlap = overlap ? 1 : 0;
    e = launch_gemm(k3, LOAD_PLAIN, STORE_SCATTER, dstatus(h), stream);
    if (e != cudaSuccess) { h->last_cuda_error = e; return SWIN_WATTN_ECUDA; }
    h->last_launches = 3;
    return SWIN_WATTN_OK;
}

int check_forward_args(const swin_wattn_s *h, const void *x, int B, int H, int W, const void *Wqkv,
                       const void *bqkv, const void *table, const float *tau, const void *Wproj, const void *bproj,
                       const void *out, bool device_io)
{
    if (!h || !x || !Wqkv || !table || !Wproj || !out) return SWIN_WATTN_EINVAL;
    if (h->mode == SWIN_WATTN_V2 && !tau) return SWIN_WATTN_EINVAL;
    int rc = check_grid(h, B, H, W);
    if (rc) return rc;
    const void *dev_ptrs[] = {Wqkv, bqkv, table, tau, Wproj, bproj};
    for (const void *p : dev_ptrs)
        if (p && !aligned16(p)) return SWIN_WATTN_EINVAL;
    if (device_io) {
        if (!aligned16(x) || !aligned16(out)) return SWIN_WATTN_EINVAL;
        const size_t bytes = (size_t)B * H * W * h->C * elem_bytes(h);
        const char *xa = (const char *)x, *oa = (const char *)out;
        if (bytes && xa < oa + bytes && oa < xa + bytes) return SWIN_WATTN_EINVAL;
    }
    return SWIN_WATTN_OK;
}

} // namespace


// ---- backward (V1) ------------------------------------------------------------

namespace {

bool overlaps(const void *a, const void *b, size_t bytes)
{
    const char *pa = (const char *)a, *pb = (const char *)b;
    return bytes && pa < pb + bytes && pb < pa + bytes;
}

// The chunked host-buffer forward on `s` (the body of swin_wattn_forward_host):
// up to h->host_chunks chunks of whole images; copy-in, compute and copy-out of different
// chunks overlap on the handle's three streams, forked from and joined back
// into `s`.  `direct`: also wait for the previous direct call's last copy.
int enqueue_host_chunks(swin_wattn_s *h, const void *x_host, int B, int H, int W, const void *Wqkv, const void *bqkv,
                        const void *table, const float *tau, const void *Wproj, const void *bproj, void *out_host,
                        cudaStream_t s, bool direct)
{
    const size_t bytes = (size_t)B * H * W * h->C * elem_bytes(h);
    cudaStream_t s_in = h->hs[0], s_run = h->hs[1], s_out = h->hs[2];
    if (cudaEventRecord(h->ev_fork, s) != cudaSuccess) return SWIN_WATTN_ECUDA;
    for (cudaStream_t st : h->hs) {
        if (cudaStreamWaitEvent(st, h->ev_fork, 0) != cudaSuccess) return SWIN_WATTN_ECUDA;
        if (direct && cudaStreamWaitEvent(st, h->ev_join, 0) != cudaSuccess) return SWIN_WATTN_ECUDA;
    }
    const int nchunks = B < h->host_chunks ? B : h->host_chunks;
    const size_t img = bytes / (size_t)B;
    int launches = 0;
    for (int c = 0; c < nchunks; ++c) {
        const int b0 = (int)((int64_t)B * c / nchunks), b1 = (int)((int64_t)B * (c + 1) / nchunks);
        const size_t off = img * (size_t)b0, len = img * (size_t)(b1 - b0);
        if (cudaMemcpyAsync((char *)h->stage_x + off, (const char *)x_host + off, len, cudaMemcpyHostToDevice,
                            s_in) != cudaSuccess ||
            cudaEventRecord(h->ev_in[c], s_in) != cudaSuccess || cudaStreamWaitEvent(s_run, h->ev_in[c], 0) != cudaSuccess)
            return SWIN_WATTN_ECUDA;
        const int rc = run_forward(h, (char *)h->stage_x + off, b1 - b0, H, W, Wqkv, bqkv, table, tau, Wproj, bproj,
                                   (char *)h->stage_out + off, s_run);
        if (rc) return rc;
        launches += h->last_launches;
        if (cudaEventRecord(h->ev_run[c], s_run) != cudaSuccess || cudaStreamWaitEvent(s_out, h->ev_run[c], 0) != cudaSuccess ||
            cudaMemcpyAsync((char *)out_host + off, (const char *)h->stage_out + off, len, cudaMemcpyDeviceToHost,
                            s_out) != cudaSuccess)
            return SWIN_WATTN_ECUDA;
    }
    h->last_launches = launches;
    // join: every stream's last work leads into s (the copy-ins precede the
    // computes, which precede the last copy-out)
    if (cudaEventRecord(h->ev_join, s_out) != cudaSuccess || cudaStreamWaitEvent(s, h->ev_join, 0) != cudaSuccess)
        return SWIN_WATTN_ECUDA;
    return SWIN_WATTN_OK;
}

} // namespace

namespace swin {

// The transformer block's use of the fused path with its LayerNorm (ln_g,
// ln_b) and residual folded in (fold 1: V1 pre-norm, 2: V2 post-norm; see
// launch_fused).  EUNSUPPORTED where this handle's forward would not take the
// fused path for the grid, or the fold does not apply to it.
int attn_forward_folded(swin_wattn_t h, const void *x, int B, int H, int W, const void *Wqkv, const void *bqkv,
                        const void *bias_table, const float *logit_scale, const void *Wproj, const void *bproj,
                        const void *ln_g, const void *ln_b, int fold, void *out, cudaStream_t stream)
{
    int rc = check_forward_args(h, x, B, H, W, Wqkv, bqkv, bias_table, logit_scale, Wproj, bproj, out, true);
    if (rc) return rc;
    if (!ln_g || !ln_b) return SWIN_WATTN_EINVAL;
    const Geom g = make_geom(B, H, W, h->C, h->M, h->shift);
    const int path = h->fp32 ? 3 : h->path_opt ? h->path_opt : choose_path(h, g.T);
    if (path != 2 || g.T >= ((int64_t)1 << 31) || !fused_fold_supported(h->M, h->C, h->heads, fold))
        return SWIN_WATTN_EUNSUPPORTED;
    h->last_launches = 0;
    if (B == 0) return SWIN_WATTN_OK;
    cudaError_t e = launch_fused((const bf16 *)x, (const bf16 *)Wqkv, (const bf16 *)bqkv, (const bf16 *)bias_table,
                                 logit_scale, (const bf16 *)Wproj, (const bf16 *)bproj, (bf16 *)out, h->mode, g,
                                 dstatus(h), h->d_err + 2, stream, (const bf16 *)ln_g, (const bf16 *)ln_b, fold,
                                 h->overlap);
    if (e != cudaSuccess) {
        h->last_cuda_error = e;
        return SWIN_WATTN_ECUDA;
    }
    h->last_launches = 1;
    return SWIN_WATTN_OK;
}

} // namespace swin

extern "C" {

int swin_wattn_create(swin_wattn_t *out, int C, int heads, int M, int shift, int mode)
{
    if (!out) return SWIN_WATTN_EINVAL;
    *out = nullptr;
    if (C <= 0 || heads <= 0 || M <= 0 || C % heads) return SWIN_WATTN_EINVAL;
    if (shift < 0 || shift >= M) return SWIN_WATTN_EINVAL;
    if (mode & ~(SWIN_WATTN_V2 | SWIN_WATTN_FP32)) return SWIN_WATTN_EINVAL;
    const bool fp32 = (mode & SWIN_WATTN_FP32) != 0;
    const int d = C / heads;
    if (!fp32 && (d != 32 || C % 32)) return SWIN_WATTN_EUNSUPPORTED;
    if (!fp32 && M > 64) return SWIN_WATTN_EUNSUPPORTED;
    if (fp32 && fp32_block_smem_bytes(M * M, C) > 200 * 1024) return SWIN_WATTN_EUNSUPPORTED;
    swin_wattn_s *h = new (std::nothrow) swin_wattn_s();
    if (!h) return SWIN_WATTN_ENOMEM;
    h->C = C; h->heads = heads; h->d = d; h->M = M; h->shift = shift;
    h->mode = mode & SWIN_WATTN_V2; h->fp32 = fp32;
    h->path_opt = 0;
    h->host_chunks = 8;
    h->overlap = 0;
    h->wait_ns = 2000000000ull;
    if (cudaGetDevice(&h->device) != cudaSuccess) { delete h; cudaGetLastError(); return SWIN_WATTN_ECUDA; }
    // [0] the error word, [2..3] the fused kernel's tile counter and CTAs done
    if (cudaMalloc(&h->d_err, 4 * sizeof(int)) != cudaSuccess) { delete h; cudaGetLastError(); return SWIN_WATTN_ENOMEM; }
    if (cudaMemset(h->d_err, 0, 4 * sizeof(int)) != cudaSuccess) { cudaFree(h->d_err); delete h; return SWIN_WATTN_ECUDA; }
    *out = h;
    return SWIN_WATTN_OK;
}

int swin_wattn_destroy(swin_wattn_t h)
{
    if (!h) return SWIN_WATTN_OK;
    cudaDeviceSynchronize();
    ws_free(&h->ws, &h->ws_bytes);
    size_t have = 0;
    ws_free(&h->stage_x, &have);
    ws_free(&h->stage_out, &have);
    ws_free(&h->bws, &h->bws_bytes);
    if (h->hs_ready) {
        for (cudaStream_t st : h->hs) cudaStreamDestroy(st);
        for (int c = 0; c < HOST_CHUNKS; ++c) {
            cudaEventDestroy(h->ev_in[c]);
            cudaEventDestroy(h->ev_run[c]);
        }
        cudaEventDestroy(h->ev_fork);
        cudaEventDestroy(h->ev_join);
        cudaEventDestroy(h->ev_done);
    }
    if (h->graph) cudaGraphExecDestroy(h->graph);
    if (h->d_err) cudaFree(h->d_err);
    delete h;
    return SWIN_WATTN_OK;
}

int swin_wattn_forward(swin_wattn_t h, const void *x, int B, int H, int W, const void *Wqkv, const void *bqkv,
                       const void *bias_table, const float *logit_scale, const void *Wproj, const void *bproj,
                       void *out, swin_stream_t stream)
{
    int rc = check_forward_args(h, x, B, H, W, Wqkv, bqkv, bias_table, logit_scale, Wproj, bproj, out, true);
    if (rc) return rc;
    rc = run_forward(h, x, B, H, W, Wqkv, bqkv, bias_table, logit_scale, Wproj, bproj, out, (cudaStream_t)stream,
                     h->overlap != 0);
    if (rc) return rc;
    return ws_check(h->ws, (cudaStream_t)stream);
}


int swin_wattn_forward_host(swin_wattn_t h, const void *x_host, int B, int H, int W, const void *Wqkv,
                            const void *bqkv, const void *bias_table, const float *logit_scale, const void *Wproj,
                            const void *bproj, void *out_host, swin_stream_t stream)
{
    int rc = check_forward_args(h, x_host, B, H, W, Wqkv, bqkv, bias_table, logit_scale, Wproj, bproj, out_host,
                                false);
    if (rc) return rc;
    const size_t bytes = (size_t)B * H * W * h->C * elem_bytes(h);
    if (bytes == 0) return SWIN_WATTN_OK;
    if (h->stage_bytes < bytes) {
        size_t have_x = h->stage_bytes, have_o = h->stage_bytes;
        rc = ws_ensure(&h->stage_x, &have_x, bytes);
        if (!rc) rc = ws_ensure(&h->stage_out, &have_o, bytes);
        if (rc) return rc;
        h->stage_bytes = bytes;
    }
    cudaStream_t s = (cudaStream_t)stream;
    if (!h->hs_ready) {
        bool ok = true;
        for (cudaStream_t &st : h->hs) ok = ok && cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) == cudaSuccess;
        for (int c = 0; c < HOST_CHUNKS; ++c) {
            ok = ok && cudaEventCreateWithFlags(&h->ev_in[c], cudaEventDisableTiming) == cudaSuccess;
            ok = ok && cudaEventCreateWithFlags(&h->ev_run[c], cudaEventDisableTiming) == cudaSuccess;
        }
        ok = ok && cudaEventCreateWithFlags(&h->ev_fork, cudaEventDisableTiming) == cudaSuccess;
        ok = ok && cudaEventCreateWithFlags(&h->ev_join, cudaEventDisableTiming) == cudaSuccess;
        ok = ok && cudaEventCreateWithFlags(&h->ev_done, cudaEventDisableTiming) == cudaSuccess;
        if (!ok) { cudaGetLastError(); return SWIN_WATTN_ECUDA; }
        h->hs_ready = true;
    }
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return SWIN_WATTN_ECUDA;
    if (cap != cudaStreamCaptureStatusNone)
        // the caller is capturing this stream: enqueue into its capture
        return enqueue_host_chunks(h, x_host, B, H, W, Wqkv, bqkv, bias_table, logit_scale, Wproj, bproj, out_host, s,
                                   false);
    // the previous call (on whatever stream) has finished with the staging buffers
    if (cudaStreamWaitEvent(s, h->ev_done, 0) != cudaSuccess) return SWIN_WATTN_ECUDA;
    // the three-kernel path's workspace for the largest chunk, before any
    // capture (no allocation may happen inside one)
    {
        const int nchunks = B < h->host_chunks ? B : h->host_chunks, bmax = (B + nchunks - 1) / nchunks;
        const int64_t Tc = (int64_t)bmax * H * W;
        const int path = h->path_opt ? h->path_opt : choose_path(h, Tc);
        if (!h->fp32 && path == 1) {
            rc = ws_ensure(&h->ws, &h->ws_bytes, (size_t)Tc * 4 * h->C * 2);
            if (rc) return rc;
        }
    }
    // the graph bakes in the call's pointers and the handle's buffers (a forward
    // on device buffers may have reallocated the workspace since)
    const void *args[11] = {x_host, Wqkv, bqkv, bias_table, logit_scale, Wproj, bproj, out_host,
                            h->ws, h->stage_x, h->stage_out};
    bool same = h->graph && h->g_B == B && h->g_H == H && h->g_W == W && h->g_path == h->path_opt &&
                h->g_chunks == h->host_chunks;
    for (int i = 0; i < 11 && same; ++i) same = h->g_args[i] == args[i];
    if (!same) {
        if (h->graph) {
            cudaGraphExecDestroy(h->graph);
            h->graph = nullptr;
        }
        cudaGraph_t graph = nullptr;
        cudaError_t ce = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
        if (ce == cudaSuccess) {
            // (the legacy default stream cannot be captured: direct enqueue below)
            rc = enqueue_host_chunks(h, x_host, B, H, W, Wqkv, bqkv, bias_table, logit_scale, Wproj, bproj, out_host,
                                     s, false);
            ce = cudaStreamEndCapture(s, &graph);
        }
        if (rc == SWIN_WATTN_OK && ce == cudaSuccess && graph && args[8] == h->ws &&
            cudaGraphInstantiate(&h->graph, graph, 0) == cudaSuccess) {
            h->g_B = B; h->g_H = H; h->g_W = W; h->g_path = h->path_opt; h->g_chunks = h->host_chunks;
            for (int i = 0; i < 11; ++i) h->g_args[i] = args[i];
            h->g_launches = h->last_launches;
        } else {
            h->graph = nullptr;
        }
        if (graph) cudaGraphDestroy(graph);
        cudaGetLastError();
        if (!h->graph) {
            // capture refused (e.g. the three-kernel workspace had to be
            // allocated first): enqueue directly; the next call captures
            rc = enqueue_host_chunks(h, x_host, B, H, W, Wqkv, bqkv, bias_table, logit_scale, Wproj, bproj, out_host,
                                     s, true);
            if (rc) return rc;
            if (cudaEventRecord(h->ev_done, s) != cudaSuccess) return SWIN_WATTN_ECUDA;
            return check_host_guards(h, s);
        }
    }
    if (cudaGraphLaunch(h->graph, s) != cudaSuccess) return SWIN_WATTN_ECUDA;
    h->last_launches = h->g_launches;
    if (cudaEventRecord(h->ev_done, s) != cudaSuccess) return SWIN_WATTN_ECUDA;
    return check_host_guards(h, s);
}

int swin_wattn_cpb_table(swin_wattn_t h, const float *W1, const float *b1, const float *W2, int hidden, void *table,
                         swin_stream_t stream)
{
    if (!h || !W1 || !W2 || !table || hidden <= 0 || hidden > 4096) return SWIN_WATTN_EINVAL;
    return cuda_status(launch_cpb_table(W1, b1, W2, hidden, h->M, h->heads, !h->fp32, table, (cudaStream_t)stream));
}

int swin_wattn_sync_status(swin_wattn_t h, swin_stream_t stream)
{
    if (!h) return SWIN_WATTN_EINVAL;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return SWIN_WATTN_ECUDA;
    int err = 0;
    if (cudaMemcpy(&err, h->d_err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return SWIN_WATTN_ECUDA;
    if (err) {
        if (cudaMemset(h->d_err, 0, sizeof(int)) != cudaSuccess) return SWIN_WATTN_ECUDA;
        if (err & ERR_TIMEOUT) return SWIN_WATTN_ETIMEOUT;
    }
    return SWIN_WATTN_OK;
}

int swin_wattn_set_option(swin_wattn_t h, int option, int64_t value)
{
    if (!h) return SWIN_WATTN_EINVAL;
    switch (option) {
    case SWIN_WATTN_OPT_PATH:
        if (value < 0 || value > 2) return SWIN_WATTN_EINVAL;
        h->path_opt = (int)value;
        return SWIN_WATTN_OK;
    case SWIN_WATTN_OPT_WAIT_LIMIT_US:
        if (value <= 0 || value > 60000000) return SWIN_WATTN_EINVAL;
        h->wait_ns = (uint64_t)value * 1000ull;
        return SWIN_WATTN_OK;
    case SWIN_WATTN_OPT_HOST_CHUNKS:
        if (value < 1 || value > HOST_CHUNKS) return SWIN_WATTN_EINVAL;
        h->host_chunks = (int)value;
        return SWIN_WATTN_OK;
    case SWIN_WATTN_OPT_OVERLAP_CALLS:
        if (value < 0 || value > 1) return SWIN_WATTN_EINVAL;
        h->overlap = (int)value;
        return SWIN_WATTN_OK;
    default:
        return SWIN_WATTN_EINVAL;
    }
}

int swin_wattn_path(swin_wattn_t h, int B, int H, int W)
{
    if (!h) return SWIN_WATTN_EINVAL;
    int rc = check_grid(h, B, H, W);
    if (rc) return rc;
    if (h->fp32) return 3;
    const int64_t T = (int64_t)B * H * W;
    const int path = h->path_opt ? h->path_opt : choose_path(h, T);
    if (path == 2 && (!fused_supported(h->M, h->C, h->heads) || T >= ((int64_t)1 << 31))) return SWIN_WATTN_EUNSUPPORTED;
    return path;
}

int swin_wattn_last_launches(swin_wattn_t h) { return h ? h->last_launches : 0; }

const char *swin_wattn_last_cuda_error(swin_wattn_t h)
{
    if (!h || h->last_cuda_error == cudaSuccess) return "no CUDA error recorded";
    return cudaGetErrorString(h->last_cuda_error);
}

const char *swin_wattn_strerror(int code)
{
    switch (code) {
    case SWIN_WATTN_OK: return "ok";
    case SWIN_WATTN_EINVAL: return "invalid argument";
    case SWIN_WATTN_EUNSUPPORTED: return "unsupported shape for the compiled kernels";
    case SWIN_WATTN_ECUDA: return "CUDA runtime error";
    case SWIN_WATTN_ENOMEM: return "device allocation failed";
    case SWIN_WATTN_ETIMEOUT: return "a kernel gave up a bounded wait";
    case SWIN_WATTN_ESCRATCH: return "intermediates exceed the fixed scratch of swin_wattn_forward_noalloc";
    case SWIN_WATTN_ECORRUPT: return "a guard band around a workspace was overwritten (SWIN_WATTN_DEBUG)";
    default: return "unknown status";
    }
}

int swin_wattn_backward(swin_wattn_t h, const void *x, int B, int H, int W, const void *Wqkv, const void *bqkv,
                        const void *bias_table, const float *logit_scale, const void *Wproj, const void *bproj,
                        const void *dy, void *dx, float *dWqkv, float *dbqkv, float *dtable, float *dlogit_scale,
                        float *dWproj, float *dbproj, swin_stream_t stream)
{
    (void)bproj;
    if (!h || !x || !Wqkv || !bias_table || !Wproj || !dy || !dx || !dWqkv || !dbqkv || !dtable || !dWproj ||
        !dbproj)
        return SWIN_WATTN_EINVAL;
    const bool v2 = h->mode == SWIN_WATTN_V2;
    if (v2 && (!logit_scale || !dlogit_scale)) return SWIN_WATTN_EINVAL;
    int rc = check_grid(h, B, H, W);
    if (rc) return rc;
    const void *ptrs[] = {x, Wqkv, bqkv, bias_table, Wproj, bproj, dy, dx, dWqkv, dbqkv, dtable, dWproj, dbproj};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return SWIN_WATTN_EINVAL;
    const int C = h->C, L = 2 * h->M - 1;
    const size_t act = (size_t)B * H * W * C * 2;
    if (overlaps(dx, x, act) || overlaps(dx, dy, act)) return SWIN_WATTN_EINVAL;
    // windows of <= 64 tokens: one kernel per (head, window pair); larger
    // windows: the forward keeps its normaliser, then key-tile units
    const bool flash = h->M * h->M > 64;
    if (h->fp32 || !(flash ? attn_flash_backward_supported(h->M, C, h->heads)
                           : attn_backward_supported(h->M, C, h->heads)))
        return SWIN_WATTN_EUNSUPPORTED;
    const Geom g = make_geom(B, H, W, C, h->M, h->shift);
    if (g.T >= ((int64_t)1 << 31)) return SWIN_WATTN_EUNSUPPORTED;
    cudaStream_t s = (cudaStream_t)stream;
    h->bw_launches = 0;
    cudaError_t e = cudaSuccess;
    auto zero = [&](float *p, size_t n) {
        if (e == cudaSuccess) e = cudaMemsetAsync(p, 0, n * sizeof(float), s);
    };
    zero(dtable, (size_t)L * L * h->heads);
    if (dlogit_scale) zero(dlogit_scale, (size_t)h->heads);
    if (B == 0) {
        zero(dbqkv, (size_t)3 * C);
        zero(dbproj, (size_t)C);
        zero(dWqkv, (size_t)3 * C * C);
        zero(dWproj, (size_t)C * C);
        return cuda_status(e);
    }
    if (e != cudaSuccess) { h->last_cuda_error = e; return SWIN_WATTN_ECUDA; }
    // workspace (bf16): attn, do [T, C]; qkv, dqkv [T, 3C]; WprojT [C, C]; WqkvT [C, 3C];
    // V2: the norms of q and k, [T, 2 heads] fp32; large windows: the
    // forward's log2 normaliser and D = do.o, [T, heads] fp32 each, and the
    // fp32 sums of dq [T, C]
    const size_t tc = (size_t)g.T * C;
    const size_t norm_bytes = v2 ? (size_t)g.T * 2 * h->heads * 4 : 0;
    const size_t flash_bytes = flash ? (size_t)g.T * 2 * h->heads * 4 + tc * 4 : 0;
    // (and the split-K partial sums of the weight gradients, fp32)
    size_t wg_bytes = wgrad_workspace_bytes(3 * C, C, g.T);
    if (wgrad_workspace_bytes(C, C, g.T) > wg_bytes) wg_bytes = wgrad_workspace_bytes(C, C, g.T);
    const size_t base_bytes = (8 * tc + 4 * (size_t)C * C) * 2 + norm_bytes + flash_bytes;
    rc = ws_ensure(&h->bws, &h->bws_bytes, base_bytes + wg_bytes);
    if (rc) return rc;
    bf16 *attn = (bf16 *)h->bws, *dO = attn + tc, *qkv = dO + tc, *dqkv = qkv + 3 * tc;
    bf16 *WpT = dqkv + 3 * tc, *WqkvT = WpT + (size_t)C * C;
    float *fws = reinterpret_cast<float *>(WqkvT + 3 * (size_t)C * C);
    float *norms = v2 ? fws : nullptr;
    if (v2) fws += (size_t)g.T * 2 * h->heads;
    float *lse = fws, *Drow = lse + (size_t)g.T * h->heads, *dq_acc = Drow + (size_t)g.T * h->heads;
    float *wg_ws = reinterpret_cast<float *>((char *)h->bws + base_bytes);
    int launches = 0;
    auto step = [&](cudaError_t r) {
        if (e == cudaSuccess) { e = r; ++launches; }
    };
    // With the overlap option the kernels after the QKV recompute start while
    // the one before them finishes.  The transposes and the recompute stay
    // ordinary launches, so every later kernel starts after both transposed
    // weights are complete (the GEMMs read their weights before they wait; the
    // attention and weight-gradient kernels read nothing before it).  The
    // large-window kernels and the dq conversion stay ordinary launches too.
    const int ov = h->overlap ? 1 : 0;
    step(launch_transpose((const bf16 *)Wproj, WpT, C, C, s));
    step(launch_transpose((const bf16 *)Wqkv, WqkvT, 3 * C, C, s));
    // window order: qkv = gather(x) Wqkv^T + bqkv, do = gather(dy) Wproj
    GemmArgs k1{};
    k1.A = (const bf16 *)x; k1.lda = C; k1.Bw = (const bf16 *)Wqkv; k1.bias = (const bf16 *)bqkv;
    k1.D = qkv; k1.ldd = 3 * C; k1.rows = g.T; k1.N = 3 * C; k1.K = C; k1.g = g;
    if (v2) { k1.norm_cols = 2 * C; k1.norms = norms; }
    step(launch_gemm(k1, LOAD_GATHER, STORE_PLAIN, dstatus(h), s));
    GemmArgs k3{};
    k3.A = (const bf16 *)dy; k3.lda = C; k3.Bw = WpT; k3.D = dO; k3.ldd = C; k3.rows = g.T; k3.N = C; k3.K = C;
    k3.g = g; k3.overlap = ov;
    step(launch_gemm(k3, LOAD_GATHER, STORE_PLAIN, dstatus(h), s));
    // o and dqkv in token order, dtable
    if (!flash) {
        step(launch_attn_backward(qkv, dO, (const bf16 *)bias_table, logit_scale, h->heads, v2 ? 1 : 0, g, attn, dqkv,
                                  dtable, norms, dlogit_scale, dstatus(h), s, ov));
    } else {
        AttnArgs k2{};
        k2.qkv = qkv; k2.attn = attn; k2.table = (const bf16 *)bias_table; k2.tau = logit_scale;
        k2.heads = h->heads; k2.mode = h->mode; k2.g = g; k2.lse = lse; k2.o_token_order = 1;
        step(launch_attention(k2, dstatus(h), s));
        zero(dq_acc, tc);
        // D, the key-tile kernel and the dq conversion: three launches
        step(launch_attn_flash_backward(qkv, dO, attn, (const bf16 *)bias_table, logit_scale, h->heads, v2 ? 1 : 0,
                                        g, lse, Drow, norms, dqkv, dq_acc, dtable, dlogit_scale, dstatus(h), s));
        launches += 2;
    }
    // dx = dqkv Wqkv (token order already)
    GemmArgs k4{};
    k4.A = dqkv; k4.lda = 3 * C; k4.Bw = WqkvT; k4.D = (bf16 *)dx; k4.ldd = C; k4.rows = g.T; k4.N = C;
    k4.K = 3 * C; k4.g = g; k4.overlap = ov;
    step(launch_gemm(k4, LOAD_PLAIN, STORE_PLAIN, dstatus(h), s));
    // dWproj = dy^T attn and dbproj, dWqkv = dqkv^T x and dbqkv: split-K tcgen05
    // GEMMs over the tokens (three launches each: partial blocks, then their
    // sum in two levels)
    step(launch_wgrad((const bf16 *)dy, C, attn, C, g.T, dWproj, dbproj, wg_ws, dstatus(h), s, ov));
    step(launch_wgrad(dqkv, 3 * C, (const bf16 *)x, C, g.T, dWqkv, dbqkv, wg_ws, dstatus(h), s, ov));
    launches += 4;
    if (e != cudaSuccess) { h->last_cuda_error = e; return SWIN_WATTN_ECUDA; }
    h->bw_launches = launches;
    return ws_check(h->bws, s);
}

int swin_wattn_backward_launches(swin_wattn_t h) { return h ? h->bw_launches : 0; }

int swin_wattn_cpb_backward(swin_wattn_t h, const float *W1, const float *b1, const float *W2, int hidden,
                            const float *dtable, float *dW1, float *db1, float *dW2, swin_stream_t stream)
{
    if (!h || !W1 || !W2 || !dtable || !dW1 || !dW2 || hidden <= 0 || hidden > 4096) return SWIN_WATTN_EINVAL;
    if (h->heads > 16) return SWIN_WATTN_EUNSUPPORTED;
    return cuda_status(launch_cpb_backward(W1, b1, W2, dtable, hidden, h->M, h->heads, dW1, db1, dW2,
                                           (cudaStream_t)stream));
}

// ---- stage hooks ------------------------------------------------------------

int swin_wattn_test_qkv(swin_wattn_t h, const void *x, int B, int H, int W, const void *Wqkv, const void *bqkv,
                        void *qkv, swin_stream_t stream)
{
    if (!h || !x || !Wqkv || !qkv || h->fp32) return SWIN_WATTN_EINVAL;
    int rc = check_grid(h, B, H, W);
    if (rc) return rc;
    if (!aligned16(x) || !aligned16(Wqkv) || !aligned16(qkv) || (bqkv && !aligned16(bqkv))) return SWIN_WATTN_EINVAL;
    if (B == 0) return SWIN_WATTN_OK;
    const Geom g = make_geom(B, H, W, h->C, h->M, h->shift);
    GemmArgs k1{};
    k1.A = (const bf16 *)x; k1.lda = h->C; k1.Bw = (const bf16 *)Wqkv; k1.bias = (const bf16 *)bqkv;
    k1.D = (bf16 *)qkv; k1.ldd = 3 * h->C; k1.rows = g.T; k1.N = 3 * h->C; k1.K = h->C; k1.g = g;
    k1.norm_cols = h->mode == SWIN_WATTN_V2 ? 2 * h->C : 0;
    return cuda_status(launch_gemm(k1, LOAD_GATHER, STORE_PLAIN, dstatus(h), (cudaStream_t)stream));
}

int swin_wattn_test_attn(swin_wattn_t h, const void *qkv, int B, int H, int W, const void *bias_table,
                         const float *logit_scale, void *attn, swin_stream_t stream)
{
    if (!h || !qkv || !bias_table || !attn || h->fp32) return SWIN_WATTN_EINVAL;
    if (h->mode == SWIN_WATTN_V2 && !logit_scale) return SWIN_WATTN_EINVAL;
    int rc = check_grid(h, B, H, W);
    if (rc) return rc;
    if (!aligned16(qkv) || !aligned16(attn)) return SWIN_WATTN_EINVAL;
    if (B == 0) return SWIN_WATTN_OK;
    AttnArgs k2{};
    k2.qkv = (const bf16 *)qkv; k2.attn = (bf16 *)attn; k2.table = (const bf16 *)bias_table; k2.tau = logit_scale;
    k2.heads = h->heads; k2.mode = h->mode; k2.g = make_geom(B, H, W, h->C, h->M, h->shift);
    return cuda_status(launch_attention(k2, dstatus(h), (cudaStream_t)stream));
}

int swin_wattn_test_proj(swin_wattn_t h, const void *attn, int B, int H, int W, const void *Wproj, const void *bproj,
                         void *out, swin_stream_t stream)
{
    if (!h || !attn || !Wproj || !out || h->fp32) return SWIN_WATTN_EINVAL;
    int rc = check_grid(h, B, H, W);
    if (rc) return rc;
    if (!aligned16(attn) || !aligned16(Wproj) || !aligned16(out) || (bproj && !aligned16(bproj))) return SWIN_WATTN_EINVAL;
    if (B == 0) return SWIN_WATTN_OK;
    const Geom g = make_geom(B, H, W, h->C, h->M, h->shift);
    GemmArgs k3{};
    k3.A = (const bf16 *)attn; k3.lda = h->C; k3.Bw = (const bf16 *)Wproj; k3.bias = (const bf16 *)bproj;
    k3.D = (bf16 *)out; k3.ldd = h->C; k3.rows = g.T; k3.N = h->C; k3.K = h->C; k3.g = g;
    return cuda_status(launch_gemm(k3, LOAD_PLAIN, STORE_SCATTER, dstatus(h), (cudaStream_t)stream));
}

int swin_wattn_test_gemm(const void *A, const void *Bw, const void *bias, void *D, int rows, int N, int K,
                         int swizzle_bytes, swin_stream_t stream)
{
    if (!A || !Bw || !D || rows < 0 || N <= 0 || K <= 0 || N % 16 || K % 16 || N > 2048) return SWIN_WATTN_EINVAL;
    if (swizzle_bytes != 0 && swizzle_bytes != 64 && swizzle_bytes != 128 && swizzle_bytes != -64 && swizzle_bytes != 1)
        return SWIN_WATTN_EINVAL;
    if (swizzle_bytes == 0 && (K % 32 || K > 128 || N > 256)) return SWIN_WATTN_EINVAL;
    if (swizzle_bytes == 1 && (K % 32 || K > 128 || N > 128)) return SWIN_WATTN_EINVAL;
    if (swizzle_bytes == -64 && (K > 128 || (N != 32 && N != 64))) return SWIN_WATTN_EINVAL;
    if (!aligned16(A) || !aligned16(Bw) || !aligned16(D) || (bias && !aligned16(bias))) return SWIN_WATTN_EINVAL;
    if (rows == 0) return SWIN_WATTN_OK;
    GemmArgs a{};
    a.A = (const bf16 *)A; a.lda = K; a.Bw = (const bf16 *)Bw; a.bias = (const bf16 *)bias;
    a.D = (bf16 *)D; a.ldd = N; a.rows = rows; a.N = N; a.K = K;
    // the hook has no handle: its error word is a private one, never read
    static int *d_err = nullptr;
    if (!d_err && cudaMalloc(&d_err, sizeof(int)) != cudaSuccess) return SWIN_WATTN_ENOMEM;
    const DeviceStatus st{d_err, 2000000000ull};
    if (swizzle_bytes == 64) return cuda_status(launch_gemm_sw64(a, st, (cudaStream_t)stream));
    if (swizzle_bytes == 0) return cuda_status(launch_gemm_ts_test(a, st, (cudaStream_t)stream));
    if (swizzle_bytes == -64) return cuda_status(launch_gemm_mn_test(a, st, (cudaStream_t)stream));
    if (swizzle_bytes == 1) {
        a.ldd = 2 * N;
        return cuda_status(launch_gemm_pair_test(a, st, (cudaStream_t)stream));
    }
    return cuda_status(launch_gemm(a, LOAD_PLAIN, STORE_PLAIN, st, (cudaStream_t)stream));
}

int swin_wattn_test_corrupt_workspace(swin_wattn_t h, int side)
{
    if (!h || (side != 0 && side != 1)) return SWIN_WATTN_EINVAL;
    return ws_test_corrupt(h->ws, side);
}

int swin_wattn_test_watchdog(swin_wattn_t h, swin_stream_t stream)
{
    if (!h) return SWIN_WATTN_EINVAL;
    return cuda_status(launch_watchdog(dstatus(h), (cudaStream_t)stream));
}

} // extern "C"
