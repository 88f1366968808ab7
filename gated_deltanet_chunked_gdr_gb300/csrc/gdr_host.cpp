// The fused call on host buffers (declared in gdr_kkt_solve.h): the inputs are
// copied to a caller-provided device workspace, the kernel runs, and the output
// is copied back, slice by slice over two streams, so that one slice's
// host-to-device copy, another's kernel and a third's device-to-host copy
// overlap.  A slice is a run of whole chunks of one sequence, so each slice is
// an independent fixed-length problem (B = 1); the result equals the one
// gdr_kkt_solve_ex gives on the whole tensor (bit for bit whenever the kernel
// takes the factored gate, i.e. every chunk's log-gate lies within 30 of its
// midpoint, since slicing can pair a tile with another partner tile, and the
// gate form is chosen per pair).  Packed sequences (cu_seqlens) go as one
// slice.
//
// Host code only: it calls the library's own entry points and the CUDA runtime
// (one cudaMemcpyAsync per tensor and slice, events for the ordering).

#include <cuda_runtime.h>

#include <mutex>
#include <stdint.h>

#include "gdr_kkt_solve.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kLanes = 2;                     // internal streams
constexpr int64_t kSliceTokenHeads = 1 << 17; // target token-heads per slice

struct Pipe {
    std::mutex mu;            // one call at a time enqueues on a device's streams
    bool ready = false;
    cudaStream_t lane[kLanes];
    cudaEvent_t start;
    cudaEvent_t done[kLanes];
};
Pipe g_pipes[kMaxDevices];

int elem_bytes(int dtype) {
    return dtype == GDR_F32 ? 4 : (dtype == GDR_BF16 || dtype == GDR_F16) ? 2 : 0;
}

int64_t round_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Workspace layout: k, g, beta (room for fp32), cu_seqlens, out, each at a
// 256-byte boundary.
struct Layout {
    int64_t k, g, beta, cu, out, total;
};

Layout layout(int k_dtype, int64_t ntok, int64_t nseq, int64_t H, int64_t K, int C, int out_dtype) {
    Layout l;
    int64_t at = 0;
    l.k = at;
    at = round_up(at + ntok * H * K * elem_bytes(k_dtype), 256);
    l.g = at;
    at = round_up(at + ntok * H * 4, 256);
    l.beta = at;
    at = round_up(at + ntok * H * 4, 256);
    l.cu = at;
    at = round_up(at + (nseq + 1) * 4, 256);
    l.out = at;
    at = round_up(at + ntok * H * C * elem_bytes(out_dtype), 256);
    l.total = at;
    return l;
}

int pipe_for_current_device(Pipe **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return GDR_ERR_DEVICE;
    }
    Pipe &p = g_pipes[dev];
    std::lock_guard<std::mutex> g(p.mu);
    if (!p.ready) {
        bool ok = cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming) == cudaSuccess;
        for (int i = 0; i < kLanes && ok; ++i)
            ok = cudaStreamCreateWithFlags(&p.lane[i], cudaStreamNonBlocking) == cudaSuccess &&
                 cudaEventCreateWithFlags(&p.done[i], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) {
            cudaGetLastError();
            return GDR_ERR_CUDA;
        }
        p.ready = true;
    }
    *out = &p;
    return GDR_OK;
}

bool valid_dtype(int d) { return d == GDR_F32 || d == GDR_BF16 || d == GDR_F16; }

}  // namespace

extern "C" {

int64_t gdr_kkt_solve_host_workspace_bytes(int k_dtype, int64_t B, int64_t T, int64_t H, int64_t K,
                                           int chunk_size, int out_dtype) {
    if (!valid_dtype(k_dtype) || !valid_dtype(out_dtype)) return GDR_ERR_DTYPE;
    if (chunk_size != 64 && chunk_size != 128) return GDR_ERR_CHUNK;
    if (B < 0 || T < 0 || H < 0 || K < 64 || K > 256 || K % 64 != 0) return GDR_ERR_SHAPE;
    if (B > (int64_t(1) << 31) || T > (int64_t(1) << 31) || H > (int64_t(1) << 24) ||
        (T > 0 && B > ((int64_t(1) << 31) - 1) / T))
        return GDR_ERR_SHAPE;
    // The larger of the fixed-length layout (B * T tokens) and the packed one
    // (T tokens, B sequences).
    const Layout l = layout(k_dtype, B * T > T ? B * T : T, B, H, K, chunk_size, out_dtype);
    return l.total;
}

int gdr_kkt_solve_host(const void *k, int k_dtype, const float *g, const void *beta, int beta_dtype,
                       const int32_t *cu_seqlens, int64_t B, int64_t T, int64_t H, int64_t K, int chunk_size,
                       int out_dtype, void *out, void *workspace, int64_t workspace_bytes, void *stream) {
    // Every argument check of the device call, without enqueuing anything: an
    // empty problem with the same types and sizes (aligned stand-in pointers).
    alignas(16) static const char stand_in[16] = {0};
    int rc = gdr_kkt_solve_ex(stand_in, k_dtype, g ? reinterpret_cast<const float *>(stand_in) : nullptr,
                              beta ? stand_in : nullptr, beta_dtype, nullptr, 0, T, H, K, chunk_size,
                              out_dtype, const_cast<char *>(stand_in), stream);
    if (rc != GDR_OK) return rc;
    if (B < 0 || T < 0 || H < 0) return GDR_ERR_SHAPE;
    if (B == 0 || T == 0 || H == 0) return GDR_OK;
    if (!k || !out || !workspace) return GDR_ERR_NULL;
    const int64_t need = gdr_kkt_solve_host_workspace_bytes(k_dtype, B, T, H, K, chunk_size, out_dtype);
    if (need < 0) return static_cast<int>(need);
    if (workspace_bytes < need) return GDR_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return GDR_ERR_ALIGN;
    if (gdr_kkt_solve_num_sms() < 0) return GDR_ERR_DEVICE;

    const int64_t ntok = cu_seqlens ? T : B * T;
    const int besz = beta ? elem_bytes(beta_dtype) : 0;
    const Layout l = layout(k_dtype, ntok, B, H, K, chunk_size, out_dtype);
    char *ws = static_cast<char *>(workspace);
    const int64_t krow = H * K * elem_bytes(k_dtype), grow = H * 4, brow = H * besz,
                  orow = H * chunk_size * elem_bytes(out_dtype);

    Pipe *pp = nullptr;
    rc = pipe_for_current_device(&pp);
    if (rc != GDR_OK) return rc;
    std::lock_guard<std::mutex> guard(pp->mu);
    cudaStream_t caller = static_cast<cudaStream_t>(stream);
    if (cudaEventRecord(pp->start, caller) != cudaSuccess) {
        cudaGetLastError();
        return GDR_ERR_CUDA;
    }
    for (int i = 0; i < kLanes; ++i)
        if (cudaStreamWaitEvent(pp->lane[i], pp->start, 0) != cudaSuccess) {
            cudaGetLastError();
            return GDR_ERR_CUDA;
        }

    // Tokens per slice: whole chunks, about kSliceTokenHeads token-heads.
    int64_t slice = round_up(kSliceTokenHeads / H > 0 ? kSliceTokenHeads / H : 1, chunk_size);
    const auto h2d = [&](int64_t off, const void *src, int64_t row0, int64_t rows, int64_t rowb,
                         cudaStream_t s) {
        return cudaMemcpyAsync(ws + off + row0 * rowb, static_cast<const char *>(src) + row0 * rowb,
                               static_cast<size_t>(rows * rowb), cudaMemcpyHostToDevice, s) == cudaSuccess;
    };
    bool ok = true;
    int n = 0;   // slices issued
    if (cu_seqlens) {
        // Packed sequences: one slice on the first lane.
        cudaStream_t s = pp->lane[0];
        ok = h2d(l.k, k, 0, T, krow, s) && (!g || h2d(l.g, g, 0, T, grow, s)) &&
             (!beta || h2d(l.beta, beta, 0, T, brow, s)) &&
             cudaMemcpyAsync(ws + l.cu, cu_seqlens, static_cast<size_t>((B + 1) * 4), cudaMemcpyHostToDevice,
                             s) == cudaSuccess;
        if (ok) {
            rc = gdr_kkt_solve_ex(ws + l.k, k_dtype, g ? reinterpret_cast<const float *>(ws + l.g) : nullptr,
                                  beta ? ws + l.beta : nullptr, beta_dtype,
                                  reinterpret_cast<const int32_t *>(ws + l.cu), B, T, H, K, chunk_size,
                                  out_dtype, ws + l.out, s);
            // Rows of real tokens only (cu[0] = 0 .. cu[B]); the rest of out is not written.
            const int64_t rows = cu_seqlens[B] < 0 ? 0 : (cu_seqlens[B] > T ? T : cu_seqlens[B]);
            ok = rc == GDR_OK &&
                 cudaMemcpyAsync(out, ws + l.out, static_cast<size_t>(rows * orow), cudaMemcpyDeviceToHost, s) ==
                     cudaSuccess;
        }
        n = 1;
    } else {
        for (int64_t b = 0; b < B && ok; ++b) {
            for (int64_t t0 = 0; t0 < T && ok; t0 += slice, ++n) {
                const int64_t rows = (T - t0 < slice) ? T - t0 : slice;
                const int64_t r0 = b * T + t0;   // first token row of the slice
                cudaStream_t s = pp->lane[n % kLanes];
                ok = h2d(l.k, k, r0, rows, krow, s) && (!g || h2d(l.g, g, r0, rows, grow, s)) &&
                     (!beta || h2d(l.beta, beta, r0, rows, brow, s));
                if (!ok) break;
                rc = gdr_kkt_solve_ex(ws + l.k + r0 * krow, k_dtype,
                                      g ? reinterpret_cast<const float *>(ws + l.g + r0 * grow) : nullptr,
                                      beta ? ws + l.beta + r0 * brow : nullptr, beta_dtype, nullptr, 1, rows, H,
                                      K, chunk_size, out_dtype, ws + l.out + r0 * orow, s);
                ok = rc == GDR_OK &&
                     cudaMemcpyAsync(static_cast<char *>(out) + r0 * orow, ws + l.out + r0 * orow,
                                     static_cast<size_t>(rows * orow), cudaMemcpyDeviceToHost, s) == cudaSuccess;
            }
        }
    }
    // The caller's stream continues after both lanes (also after a failure, so
    // nothing the caller enqueues later overtakes work already issued).
    for (int i = 0; i < kLanes; ++i)
        if (cudaEventRecord(pp->done[i], pp->lane[i]) != cudaSuccess ||
            cudaStreamWaitEvent(caller, pp->done[i], 0) != cudaSuccess)
            ok = false;
    if (!ok) {
        cudaGetLastError();
        return rc != GDR_OK ? rc : GDR_ERR_CUDA;
    }
    return GDR_OK;
}

}  // extern "C"
