// C-ABI entry points: argument validation, kernel choice, status word.
#include <atomic>
#include <cstring>
#include <mutex>

#include "mmq_internal.h"

namespace {

__device__ int g_status_word;   // one per device (module globals are per context)

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_status_addr[kMaxDevices];       // device address of g_status_word
signed char g_arch_ok[kMaxDevices];    // 0 unknown, 1 sm_103, -1 other

thread_local int t_inject_timeout = 0;
std::atomic<int> g_programmatic_launch{0};

int current_device(int* dev) {
    if (cudaGetDevice(dev) != cudaSuccess) { cudaGetLastError(); return MMQ_ERR_CUDA; }
    if (*dev < 0 || *dev >= kMaxDevices) return MMQ_ERR_DEVICE;
    return MMQ_OK;
}

int check_device() {
    int dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_arch_ok[dev] == 0) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return MMQ_ERR_CUDA;
        }
        g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    }
    return g_arch_ok[dev] == 1 ? MMQ_OK : MMQ_ERR_DEVICE;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int check_q8(const mmq_q8_1_t& aq) {
    if (!aq.qs || !aq.da || !aq.sa) return MMQ_ERR_ARG;
    if (!aligned16(aq.qs) || !aligned16(aq.da) || !aligned16(aq.sa)) return MMQ_ERR_ALIGN;
    return MMQ_OK;
}

int check_gemm_args(const mmq_q8_1_t& aq, const void* w, const void* out, int64_t M,
                    int64_t N, int64_t K) {
    int rc = check_q8(aq);
    if (rc) return rc;
    if (!w || !out) return MMQ_ERR_ARG;
    if (M < 1 || N < 1 || K < 256 || (K % 256) != 0 || (N % 4) != 0) return MMQ_ERR_ARG;
    // Coordinates fed to the kernels and tensor maps are 32-bit.
    if (M > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 31) - 1)
        return MMQ_ERR_ARG;
    if (!aligned16(w) || !aligned16(out)) return MMQ_ERR_ALIGN;
    return check_device();
}

int from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return MMQ_OK;
    cudaGetLastError();
    return MMQ_ERR_CUDA;
}

}  // namespace

namespace mmq {

bool programmatic_launch_enabled() { return g_programmatic_launch.load(std::memory_order_relaxed) != 0; }

int* status_word_ptr() {
    int dev;
    if (current_device(&dev)) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_status_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_status_addr[dev] = static_cast<int*>(p);
    }
    return g_status_addr[dev];
}

}  // namespace mmq

extern "C" {

size_t mmq_q8_1_bytes(int64_t M, int64_t K) {
    if (M < 1 || K < 32 || (K % 32) != 0) return 0;
    auto up = [](size_t b) { return (b + 255) & ~size_t(255); };
    const size_t nb = size_t(M) * size_t(K / 32);
    return up(size_t(M) * size_t(K)) + up(nb * 4) + up(nb * 4);
}

int mmq_q8_1_view(void* buf, int64_t M, int64_t K, mmq_q8_1_t* out) {
    if (!buf || !out || mmq_q8_1_bytes(M, K) == 0) return MMQ_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(buf) & 255) return MMQ_ERR_ALIGN;
    auto up = [](size_t b) { return (b + 255) & ~size_t(255); };
    const size_t nb = size_t(M) * size_t(K / 32);
    char* p = static_cast<char*>(buf);
    out->qs = reinterpret_cast<int8_t*>(p);
    out->da = reinterpret_cast<float*>(p + up(size_t(M) * size_t(K)));
    out->sa = reinterpret_cast<int32_t*>(p + up(size_t(M) * size_t(K)) + up(nb * 4));
    return MMQ_OK;
}

int mmq_quantize_q8_1(const float* x, int64_t M, int64_t K, mmq_q8_1_t aq, void* stream) {
    if (!x) return MMQ_ERR_ARG;
    int rc = check_q8(aq);
    if (rc) return rc;
    if (M < 1 || K < 32 || (K % 32) != 0) return MMQ_ERR_ARG;
    if (M > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 31) - 1) return MMQ_ERR_ARG;
    if (!aligned16(x)) return MMQ_ERR_ALIGN;
    if ((rc = check_device())) return rc;
    return from_cuda(mmq::launch_quantize_q8_1(x, M, K, aq, static_cast<cudaStream_t>(stream)));
}

size_t mmq_q8_1_tcop_bytes(int64_t M, int64_t K) {
    if (M < 1 || K < 256 || (K % 256) != 0) return 0;
    if (M > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 31) - 1) return 0;
    return mmq::tcop_layout(M, K).bytes;
}

int mmq_quantize_q8_1_tcop(const float* x, int64_t M, int64_t K, mmq_q8_1_t aq, void* tcop, void* stream) {
    if (!x || !tcop) return MMQ_ERR_ARG;
    int rc = check_q8(aq);
    if (rc) return rc;
    if (mmq_q8_1_tcop_bytes(M, K) == 0) return MMQ_ERR_ARG;
    if (!aligned16(x)) return MMQ_ERR_ALIGN;
    if (reinterpret_cast<uintptr_t>(tcop) & 255) return MMQ_ERR_ALIGN;
    if ((rc = check_device())) return rc;
    return from_cuda(mmq::launch_quantize_q8_1_tcop(x, M, K, aq, tcop, static_cast<cudaStream_t>(stream)));
}

size_t mmq_q4K_bytes(int64_t N, int64_t K) {
    if (N < 1 || K < 256 || (K % 256) != 0) return 0;
    return size_t(N) * size_t(K / 256) * 144;
}

// The automatic kernel choice (shape only): few tokens -> weight streaming,
// else the tcgen05 kernel.
static int auto_path(int64_t M, int64_t N) {
    (void)N;
    return M <= mmq::kSmallMMax ? MMQ_PATH_SMALL_M : MMQ_PATH_TC;
}

static bool known_path(int path) {
    return path == MMQ_PATH_AUTO || path == MMQ_PATH_MMA_S8 || path == MMQ_PATH_TC || path == MMQ_PATH_SMALL_M;
}

static int run_gemm(mmq_q8_1_t aq, const uint8_t* w, float* C, int32_t* S, int64_t M,
                    int64_t N, int64_t K, int path, cudaStream_t s,
                    mmq_q8_1_t q8out = mmq_q8_1_t{nullptr, nullptr, nullptr}, bool dump_scaled = false) {
    int* status = mmq::status_word_ptr();
    if (!status) return MMQ_ERR_CUDA;
    if (path == MMQ_PATH_AUTO) path = auto_path(M, N);
    switch (path) {
        case MMQ_PATH_MMA_S8:
            return from_cuda(mmq::launch_gemm_mma_s8(aq, w, C, S, M, N, K, status, s));
        case MMQ_PATH_TC: {
            int rc = mmq::tc_gemm_check_resources();
            if (rc) return rc;
            const int inject = t_inject_timeout;
            t_inject_timeout = 0;
            return from_cuda(mmq::launch_gemm_tc(aq, w, C, q8out, S, M, N, K, status, inject, s, false,
                                                 dump_scaled));
        }
        case MMQ_PATH_SMALL_M:
            if (M > mmq::kSmallMMax) return MMQ_ERR_ARG;
            if (S)
                return from_cuda(mmq::launch_gemm_small_m(aq, w, nullptr, M, N, K, status, s,
                                                          mmq_q8_1_t{nullptr, nullptr, nullptr}, mmq::kSmallDump, S));
            return from_cuda(mmq::launch_gemm_small_m(aq, w, C, M, N, K, status, s));
        default:
            return MMQ_ERR_ARG;
    }
}

int mmq_q4K_gemm(mmq_q8_1_t aq, const uint8_t* bq4k, float* C, int64_t M, int64_t N,
                 int64_t K, void* stream) {
    return mmq_q4K_gemm_path(aq, bq4k, C, M, N, K, MMQ_PATH_AUTO, stream);
}

static int gemm_auto(mmq_q8_1_t aq, const uint8_t* w, float* C, int64_t M, int64_t N, int64_t K,
                     cudaStream_t s) {
    return run_gemm(aq, w, C, nullptr, M, N, K, MMQ_PATH_AUTO, s);
}

size_t mmq_q4K_gemm_host_workspace(int64_t M, int64_t N, int64_t K) {
    if (M < 1 || N < 1 || K < 256 || (K % 256) != 0 || (N % 4) != 0) return 0;
    if (M > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 31) - 1) return 0;
    return mmq::host_workspace_bytes(M, N, K);
}

int mmq_q4K_gemm_host(const float* x_host, const uint8_t* bq4k, float* C_host, int64_t M, int64_t N, int64_t K,
                      void* workspace, size_t workspace_bytes, void* stream) {
    if (!x_host || !bq4k || !C_host || !workspace) return MMQ_ERR_ARG;
    const size_t need = mmq_q4K_gemm_host_workspace(M, N, K);
    if (need == 0 || workspace_bytes < need) return MMQ_ERR_ARG;
    if (!aligned16(bq4k) || (reinterpret_cast<uintptr_t>(workspace) & 255)) return MMQ_ERR_ALIGN;
    int rc = check_device();
    if (rc) return rc;
    return mmq::gemm_host(x_host, bq4k, C_host, M, N, K, workspace, static_cast<cudaStream_t>(stream), gemm_auto);
}

int mmq_q4K_gemm_host_noalloc(const float* x_host, const uint8_t* bq4k, float* C_host, int64_t M, int64_t N,
                              int64_t K, void* stream) {
    if (!x_host || !bq4k || !C_host) return MMQ_ERR_ARG;
    const size_t need = mmq_q4K_gemm_host_workspace(M, N, K);
    if (need == 0 || need > MMQ_HOST_NOALLOC_SCRATCH_BYTES) return MMQ_ERR_ARG;
    if (!aligned16(bq4k)) return MMQ_ERR_ALIGN;
    int rc = check_device();
    if (rc) return rc;
    void* scratch = nullptr;
    if ((rc = mmq::host_noalloc_scratch(&scratch))) return rc;
    return mmq::gemm_host(x_host, bq4k, C_host, M, N, K, scratch, static_cast<cudaStream_t>(stream), gemm_auto);
}

int mmq_q4K_gemm_launches(int64_t M, int64_t N, int64_t K, int path) {
    if (!known_path(path)) return MMQ_ERR_ARG;
    if (M < 1 || N < 1 || K < 256 || (K % 256) != 0 || (N % 4) != 0) return MMQ_ERR_ARG;
    if (M > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 31) - 1)
        return MMQ_ERR_ARG;
    if (path == MMQ_PATH_SMALL_M && M > mmq::kSmallMMax) return MMQ_ERR_ARG;
    int rc = check_device();
    if (rc) return rc;
    if (path == MMQ_PATH_AUTO) path = auto_path(M, N);
    if (path != MMQ_PATH_TC && path != MMQ_PATH_SMALL_M) return 1;
    const int n = path == MMQ_PATH_TC ? mmq::tc_gemm_launch_count(M, N, K) : mmq::small_m_launch_count(M, N, K);
    return n < 0 ? MMQ_ERR_CUDA : n;
}

int mmq_q4K_gemm_path(mmq_q8_1_t aq, const uint8_t* bq4k, float* C, int64_t M, int64_t N,
                      int64_t K, int path, void* stream) {
    if (!known_path(path)) return MMQ_ERR_ARG;
    if (path == MMQ_PATH_SMALL_M && M > mmq::kSmallMMax) return MMQ_ERR_ARG;
    int rc = check_gemm_args(aq, bq4k, C, M, N, K);
    if (rc) return rc;
    return run_gemm(aq, bq4k, C, nullptr, M, N, K, path, static_cast<cudaStream_t>(stream));
}

int mmq_q4K_gemm_tcop(const void* tcop, const uint8_t* bq4k, float* C, int64_t M, int64_t N, int64_t K,
                      void* stream) {
    if (!tcop || !bq4k || !C) return MMQ_ERR_ARG;
    if (mmq_q8_1_tcop_bytes(M, K) == 0 || N < 1 || (N % 4) != 0 || N > (int64_t(1) << 31) - 1) return MMQ_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(tcop) & 255) || !aligned16(bq4k) || !aligned16(C)) return MMQ_ERR_ALIGN;
    int rc = check_device();
    if (rc) return rc;
    if ((rc = mmq::sb_gemm_check_resources())) return rc;
    int* status = mmq::status_word_ptr();
    if (!status) return MMQ_ERR_CUDA;
    const int inject = t_inject_timeout;
    t_inject_timeout = 0;
    return from_cuda(mmq::launch_gemm_sb(tcop, bq4k, C, M, N, K, status, inject, static_cast<cudaStream_t>(stream)));
}

int mmq_q4K_gemm_q8_1(mmq_q8_1_t aq, const uint8_t* bq4k, float* C, mmq_q8_1_t out, int64_t M,
                      int64_t N, int64_t K, void* stream) {
    int rc = check_q8(out);
    if (rc) return rc;
    if (N % 32 != 0) return MMQ_ERR_ARG;
    const bool small = M <= mmq::kSmallMMax;
    rc = check_gemm_args(aq, bq4k, C ? static_cast<const void*>(C) : static_cast<const void*>(out.qs), M, N, K);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (small) {   // one few-token kernel with the quantizing epilogue
        int* status = mmq::status_word_ptr();
        if (!status) return MMQ_ERR_CUDA;
        return from_cuda(mmq::launch_gemm_small_m(aq, bq4k, C, M, N, K, status, s, out, 1));
    }
    return run_gemm(aq, bq4k, C, nullptr, M, N, K, MMQ_PATH_TC, s, out);
}

int mmq_q4K_gemm_swiglu_q8_1(mmq_q8_1_t aq, const uint8_t* bq4k_gu, float* hf, mmq_q8_1_t out, int64_t M,
                             int64_t F, int64_t K, void* stream) {
    int rc = check_q8(out);
    if (rc) return rc;
    if (F < 32 || (F % 32) != 0 || F > (int64_t(1) << 30)) return MMQ_ERR_ARG;
    if ((rc = check_gemm_args(aq, bq4k_gu, out.qs, M, 2 * F, K))) return rc;
    if (hf && !aligned16(hf)) return MMQ_ERR_ALIGN;
    if (M <= mmq::kSmallMMax) {   // one few-token kernel, SwiGLU and q8_1 in its epilogue
        int* status = mmq::status_word_ptr();
        if (!status) return MMQ_ERR_CUDA;
        return from_cuda(mmq::launch_gemm_small_m(aq, bq4k_gu, hf, M, 2 * F, K, status,
                                                  static_cast<cudaStream_t>(stream), out, 2));
    }
    if ((rc = mmq::tc_gemm_check_resources())) return rc;
    int* status = mmq::status_word_ptr();
    if (!status) return MMQ_ERR_CUDA;
    const int inject = t_inject_timeout;
    t_inject_timeout = 0;
    return from_cuda(mmq::launch_gemm_tc(aq, bq4k_gu, hf, out, nullptr, M, 2 * F, K, status, inject,
                                         static_cast<cudaStream_t>(stream), true));
}

int mmq_interleave_rows_q4K(const uint8_t* gate, const uint8_t* up, uint8_t* out, int64_t F, int64_t K,
                            void* stream) {
    if (!gate || !up || !out) return MMQ_ERR_ARG;
    if (F < 1 || K < 256 || (K % 256) != 0 || F > (int64_t(1) << 30) || K > (int64_t(1) << 31) - 1)
        return MMQ_ERR_ARG;
    int rc = check_device();
    if (rc) return rc;
    const size_t pitch = size_t(K / 256) * 144;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpy2DAsync(out, 2 * pitch, gate, pitch, pitch, size_t(F), cudaMemcpyDefault, s);
    if (e == cudaSuccess)
        e = cudaMemcpy2DAsync(out + pitch, 2 * pitch, up, pitch, pitch, size_t(F), cudaMemcpyDefault, s);
    return from_cuda(e);
}

int mmq_q4K_block_dots(mmq_q8_1_t aq, const uint8_t* bq4k, int32_t* S, int64_t M, int64_t N,
                       int64_t K, int path, void* stream) {
    if (!known_path(path)) return MMQ_ERR_ARG;
    if (path == MMQ_PATH_SMALL_M && M > mmq::kSmallMMax) return MMQ_ERR_ARG;
    int rc = check_gemm_args(aq, bq4k, S, M, N, K);
    if (rc) return rc;
    return run_gemm(aq, bq4k, nullptr, S, M, N, K, path, static_cast<cudaStream_t>(stream));
}

int mmq_q4K_scaled_block_dots(mmq_q8_1_t aq, const uint8_t* bq4k, int32_t* S, int64_t M, int64_t N,
                              int64_t K, void* stream) {
    int rc = check_gemm_args(aq, bq4k, S, M, N, K);
    if (rc) return rc;
    return run_gemm(aq, bq4k, nullptr, S, M, N, K, MMQ_PATH_TC, static_cast<cudaStream_t>(stream),
                    mmq_q8_1_t{nullptr, nullptr, nullptr}, true);
}

int mmq_dequantize_q4K_f16(const uint8_t* bq4k, uint16_t* wh, int64_t N, int64_t K, void* stream) {
    if (!bq4k || !wh) return MMQ_ERR_ARG;
    if (N < 1 || K < 256 || (K % 256) != 0) return MMQ_ERR_ARG;
    if (N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 31) - 1 || N * (K / 64) > (int64_t(1) << 36))
        return MMQ_ERR_ARG;
    if (!aligned16(bq4k) || !aligned16(wh)) return MMQ_ERR_ALIGN;
    int rc = check_device();
    if (rc) return rc;
    return from_cuda(mmq::launch_dequantize_q4K_f16(bq4k, wh, N, K, static_cast<cudaStream_t>(stream)));
}

int mmq_convert_f32_f16(const float* x, uint16_t* xh, int64_t n, void* stream) {
    if (!x || !xh) return MMQ_ERR_ARG;
    if (n < 4 || (n % 4) != 0 || n > (int64_t(1) << 38)) return MMQ_ERR_ARG;
    if (!aligned16(x) || !aligned16(xh)) return MMQ_ERR_ALIGN;
    int rc = check_device();
    if (rc) return rc;
    return from_cuda(mmq::launch_convert_f16(x, xh, n, static_cast<cudaStream_t>(stream)));
}

int mmq_gemm_f16(const uint16_t* A, const uint16_t* B, float* C, int64_t M, int64_t N, int64_t K,
                 void* stream) {
    if (!A || !B || !C) return MMQ_ERR_ARG;
    if (M < 1 || N < 1 || K < 64 || (K % 64) != 0 || (N % 4) != 0) return MMQ_ERR_ARG;
    if (M > (int64_t(1) << 31) - 1 || N > (int64_t(1) << 31) - 1 || K > (int64_t(1) << 31) - 1)
        return MMQ_ERR_ARG;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C)) return MMQ_ERR_ALIGN;
    int rc = check_device();
    if (rc) return rc;
    if ((rc = mmq::dense_gemm_check_resources())) return rc;
    int* status = mmq::status_word_ptr();
    if (!status) return MMQ_ERR_CUDA;
    return from_cuda(mmq::launch_gemm_f16(A, B, C, M, N, K, status, static_cast<cudaStream_t>(stream)));
}

size_t mmq_q6K_dev_bytes(int64_t N, int64_t K) {
    if (N < 1 || K < 256 || (K % 256) != 0) return 0;
    return size_t(N) * size_t(K / 256) * 224;
}

int mmq_repack_q6K(const uint8_t* src, uint8_t* dst, int64_t N, int64_t K, void* stream) {
    if (!src || !dst) return MMQ_ERR_ARG;
    if (N < 1 || K < 256 || (K % 256) != 0 || N * (K / 256) > (int64_t(1) << 34)) return MMQ_ERR_ARG;
    if (!aligned16(dst)) return MMQ_ERR_ALIGN;
    int rc = check_device();
    if (rc) return rc;
    return from_cuda(mmq::launch_repack_q6K(src, dst, N, K, static_cast<cudaStream_t>(stream)));
}

// The q6_K kernel family for M tokens: the dot-product kernel for a few,
// the tcgen05 kernel above that.
static int q6k_auto_path(int64_t M) { return M <= mmq::kQ6GemvMax ? MMQ_PATH_SMALL_M : MMQ_PATH_TC; }

int mmq_q6K_gemm_path(mmq_q8_1_t aq, const uint8_t* bq6k_dev, float* C, int64_t M, int64_t N, int64_t K,
                      int path, void* stream) {
    if (!known_path(path)) return MMQ_ERR_ARG;
    int rc = check_gemm_args(aq, bq6k_dev, C, M, N, K);
    if (rc) return rc;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (path == MMQ_PATH_AUTO) path = q6k_auto_path(M);
    switch (path) {
        case MMQ_PATH_SMALL_M:
            if (M > mmq::kQ6GemvMax) return MMQ_ERR_ARG;
            return from_cuda(mmq::launch_gemm_q6k(aq, bq6k_dev, C, nullptr, M, N, K, s));
        case MMQ_PATH_MMA_S8:
            return from_cuda(mmq::launch_gemm_q6k(aq, bq6k_dev, C, nullptr, M, N, K, s, false));
        default: {   // MMQ_PATH_TC
            if ((rc = mmq::q6k_tc_check_resources())) return rc;
            int* status = mmq::status_word_ptr();
            if (!status) return MMQ_ERR_CUDA;
            const int inject = t_inject_timeout;
            t_inject_timeout = 0;
            return from_cuda(mmq::launch_gemm_q6k_tc(aq, bq6k_dev, C, nullptr, M, N, K, status, inject, s));
        }
    }
}

int mmq_q6K_gemm(mmq_q8_1_t aq, const uint8_t* bq6k_dev, float* C, int64_t M, int64_t N, int64_t K,
                 void* stream) {
    return mmq_q6K_gemm_path(aq, bq6k_dev, C, M, N, K, MMQ_PATH_AUTO, stream);
}

int mmq_q6K_scaled_block_dots(mmq_q8_1_t aq, const uint8_t* bq6k_dev, int32_t* S, int64_t M, int64_t N,
                              int64_t K, void* stream) {
    int rc = check_gemm_args(aq, bq6k_dev, S, M, N, K);
    if (rc) return rc;
    if ((rc = mmq::q6k_tc_check_resources())) return rc;
    int* status = mmq::status_word_ptr();
    if (!status) return MMQ_ERR_CUDA;
    return from_cuda(mmq::launch_gemm_q6k_tc(aq, bq6k_dev, nullptr, S, M, N, K, status, 0,
                                             static_cast<cudaStream_t>(stream)));
}

int mmq_q6K_gemm_launches(int64_t M, int64_t N, int64_t K, int path) {
    if (!known_path(path) || M < 1 || N < 1 || K < 256 || (K % 256) != 0) return MMQ_ERR_ARG;
    if (path == MMQ_PATH_AUTO) path = q6k_auto_path(M);
    if (path == MMQ_PATH_SMALL_M && M > mmq::kQ6GemvMax) return MMQ_ERR_ARG;
    if (path != MMQ_PATH_TC) return 1;
    const int n = mmq::q6k_tc_launch_count(M, N, K);
    return n < 0 ? MMQ_ERR_CUDA : n;
}

int mmq_q6K_block_dots(mmq_q8_1_t aq, const uint8_t* bq6k_dev, int32_t* S, int64_t M, int64_t N, int64_t K,
                       void* stream) {
    int rc = check_gemm_args(aq, bq6k_dev, S, M, N, K);
    if (rc) return rc;
    return from_cuda(mmq::launch_gemm_q6k(aq, bq6k_dev, nullptr, S, M, N, K, static_cast<cudaStream_t>(stream)));
}

int mmq_status(void* stream) {
    int* p = mmq::status_word_ptr();
    if (!p) return MMQ_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int v = 0;
    const int zero = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) { cudaGetLastError(); return MMQ_ERR_CUDA; }
    if (cudaMemcpyAsync(&v, p, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(p, &zero, sizeof(int), cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return MMQ_ERR_CUDA;
    }
    return v;
}

const char* mmq_strerror(int code) {
    switch (code) {
        case MMQ_OK: return "ok";
        case MMQ_ERR_ARG: return "invalid argument (null pointer, size or value range)";
        case MMQ_ERR_ALIGN: return "pointer not 16-byte aligned";
        case MMQ_ERR_DEVICE: return "current device is not sm_103 (GB300)";
        case MMQ_ERR_RESOURCE: return "shared/tensor memory budget exceeded; launch refused";
        case MMQ_ERR_CUDA: return "CUDA runtime error";
        case MMQ_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait timed out; output invalid";
        default: return "unknown error code";
    }
}

void mmq_debug_inject_timeout(int enable) { t_inject_timeout = enable ? 1 : 0; }

int mmq_debug_force_gemv_split(int ks) { return mmq::set_force_gemv_split(ks); }

void mmq_set_programmatic_launch(int enable) { g_programmatic_launch.store(enable ? 1 : 0); }

}  // extern "C"
