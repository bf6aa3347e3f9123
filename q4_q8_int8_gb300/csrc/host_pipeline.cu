// The prepass + GEMM with activations and result in host memory: the rows are
// cut into chunks, and chunk i+1's host-to-device copy, chunk i's prepass
// and GEMM and chunk i-1's device-to-host copy run at the same time on three
// streams (the caller's for the kernels, two of the library's for the two
// copy directions), ordered by events.  Device workspace is the caller's:
// two x chunks, one q8_1 chunk, two C chunks.
#include <mutex>

#include "mmq_internal.h"

namespace {

constexpr int kMaxDevices = 64;

struct HostPipe {   // per device, created on first use and kept for the process
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, in_done[2] = {}, comp_done[2] = {}, out_done[2] = {};
};

std::mutex g_pipe_mu;   // held while a pipeline is enqueued: one at a time per process
HostPipe g_pipe[kMaxDevices];

cudaError_t pipe_for(int dev, HostPipe** out) {
    HostPipe& p = g_pipe[dev];
    if (!p.in) {
        cudaError_t e = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming);
        for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
            e = cudaEventCreateWithFlags(&p.in_done[b], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.comp_done[b], cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.out_done[b], cudaEventDisableTiming);
        }
        if (e != cudaSuccess) {
            p = HostPipe{};   // handles created so far are leaked, not reused half-made
            return e;
        }
    }
    *out = &p;
    return cudaSuccess;
}

size_t up256(size_t b) { return (b + 255) & ~size_t(255); }

// The fixed device workspace of mmq_q4K_gemm_host_noalloc.  Every device on
// which the library's code is loaded holds it until the process exits.  In
// host code the name is only a host-side stand-in for the array; its device
// address comes from cudaGetSymbolAddress, looked up once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MMQ_HOST_NOALLOC_SCRATCH_BYTES];
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices];

}  // namespace

namespace mmq {

int host_noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return MMQ_ERR_DEVICE;
    }
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {   // first call on this device (it is the current one)
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return MMQ_ERR_CUDA;
        }
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return MMQ_OK;
}

int64_t host_chunk_rows(int64_t M) {
    if (M <= 256) return M;
    const int64_t quarter = (M + 3) / 4;
    const int64_t r = (quarter + 127) / 128 * 128;
    return r < 256 ? 256 : r;
}

size_t host_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    const size_t mc = size_t(host_chunk_rows(M));
    const size_t nb = mc * size_t(K / 32);
    return 2 * up256(mc * size_t(K) * 4) + up256(mc * size_t(K)) + 2 * up256(nb * 4) + 2 * up256(mc * size_t(N) * 4);
}

int gemm_host(const float* x_host, const uint8_t* w, float* C_host, int64_t M, int64_t N, int64_t K, void* ws,
              cudaStream_t s0, GemmFn gemm) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return MMQ_ERR_DEVICE;
    }
    const int64_t Mc = host_chunk_rows(M);
    const size_t xbytes = up256(size_t(Mc) * size_t(K) * 4), cbytes = up256(size_t(Mc) * size_t(N) * 4);
    const size_t nb = size_t(Mc) * size_t(K / 32);
    char* p = static_cast<char*>(ws);
    float* xb[2] = {reinterpret_cast<float*>(p), reinterpret_cast<float*>(p + xbytes)};
    p += 2 * xbytes;
    mmq_q8_1_t q8;
    q8.qs = reinterpret_cast<int8_t*>(p);
    p += up256(size_t(Mc) * size_t(K));
    q8.da = reinterpret_cast<float*>(p);
    p += up256(nb * 4);
    q8.sa = reinterpret_cast<int32_t*>(p);
    p += up256(nb * 4);
    float* cb[2] = {reinterpret_cast<float*>(p), reinterpret_cast<float*>(p + cbytes)};

    std::lock_guard<std::mutex> lk(g_pipe_mu);
    HostPipe* hp = nullptr;
    cudaError_t e = pipe_for(dev, &hp);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return MMQ_ERR_CUDA;
    }
    auto ck = [&](cudaError_t r) {
        if (e == cudaSuccess) e = r;
    };
    // the copies start after everything already queued on the caller's stream
    ck(cudaEventRecord(hp->start, s0));
    ck(cudaStreamWaitEvent(hp->in, hp->start, 0));
    ck(cudaStreamWaitEvent(hp->out, hp->start, 0));
    const int64_t nchunks = (M + Mc - 1) / Mc;
    for (int64_t i = 0; i < nchunks && e == cudaSuccess; ++i) {
        const int b = int(i & 1);
        const int64_t r0 = i * Mc, mc = (M - r0) < Mc ? (M - r0) : Mc;
        // in: x buffer b is free once chunk i-2's prepass has read it
        if (i >= 2) ck(cudaStreamWaitEvent(hp->in, hp->comp_done[b], 0));
        ck(cudaMemcpyAsync(xb[b], x_host + r0 * K, size_t(mc) * size_t(K) * 4, cudaMemcpyHostToDevice, hp->in));
        ck(cudaEventRecord(hp->in_done[b], hp->in));
        // kernels: C buffer b is free once chunk i-2's result has left
        ck(cudaStreamWaitEvent(s0, hp->in_done[b], 0));
        if (i >= 2) ck(cudaStreamWaitEvent(s0, hp->out_done[b], 0));
        if (e != cudaSuccess) break;
        ck(launch_quantize_q8_1(xb[b], mc, K, q8, s0));
        if (e != cudaSuccess) break;
        const int rc = gemm(q8, w, cb[b], mc, N, K, s0);
        if (rc != MMQ_OK) {
            cudaGetLastError();
            // join both copy streams back into the caller's stream, so that
            // work queued there later (or a graph capture) stays ordered
            // after the copies already issued
            for (cudaStream_t cs : {hp->in, hp->out})
                if (cudaEventRecord(hp->start, cs) == cudaSuccess) cudaStreamWaitEvent(s0, hp->start, 0);
            cudaGetLastError();
            return rc;
        }
        ck(cudaEventRecord(hp->comp_done[b], s0));
        // out
        ck(cudaStreamWaitEvent(hp->out, hp->comp_done[b], 0));
        ck(cudaMemcpyAsync(C_host + r0 * N, cb[b], size_t(mc) * size_t(N) * 4, cudaMemcpyDeviceToHost, hp->out));
        ck(cudaEventRecord(hp->out_done[b], hp->out));
    }
    // the caller's stream is ordered after the last copies of both buffers
    for (int b = 0; b < 2 && b < nchunks && e == cudaSuccess; ++b) ck(cudaStreamWaitEvent(s0, hp->out_done[b], 0));
    if (e != cudaSuccess) {
        cudaGetLastError();
        for (cudaStream_t cs : {hp->in, hp->out})   // best effort: keep the caller's stream joined
            if (cudaEventRecord(hp->start, cs) == cudaSuccess) cudaStreamWaitEvent(s0, hp->start, 0);
        cudaGetLastError();
        return MMQ_ERR_CUDA;
    }
    return MMQ_OK;
}

}  // namespace mmq
