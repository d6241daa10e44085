// C ABI of libqoq.so: argument validation, workspace planning and launches.
// Declarations and the full contract of each entry point: include/qoq.h.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/qoq.h"
#include "qoq_internal.h"

namespace {

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// QOQ_OK when the current device is one the library serves (its ordinal is
// below qoq::kMaxDevices); checked before any planning or launch.
int check_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QOQ_ERR_CUDA;
    return (dev >= 0 && dev < qoq::kMaxDevices) ? QOQ_OK : QOQ_ERR_UNSUPPORTED;
}

int num_sms_current_device() {
    static std::mutex mu;
    static int cache[qoq::kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= qoq::kMaxDevices) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] > 0) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
    return n;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? QOQ_OK : QOQ_ERR_CUDA; }

int check_gemm_shape(int M, int N, int K, int group) {
    if (M <= 0 || N <= 0 || K <= 0) return QOQ_ERR_INVALID_ARG;
    if (group != 0 && group != 128) return QOQ_ERR_UNSUPPORTED;
    if (N % 128 != 0 || K % 128 != 0) return QOQ_ERR_UNSUPPORTED;
    if (N / 128 > 65535) return QOQ_ERR_UNSUPPORTED;
    return QOQ_OK;
}

int check_options(const qoq_gemm_options *opt) {
    if (!opt) return QOQ_OK;
    const int bt = opt->tokens_per_tile;
    if (bt != 0 && bt != 16 && bt != 32 && bt != 64 && bt != 128) return QOQ_ERR_UNSUPPORTED;
    if (opt->num_ctas < 0 || opt->num_ctas > 65536) return QOQ_ERR_UNSUPPORTED;
    if (opt->kernel < 0 || opt->kernel > 3) return QOQ_ERR_UNSUPPORTED;
    if (opt->flags & ~(QOQ_LAUNCH_OVERLAP | QOQ_PLAN_RULES)) return QOQ_ERR_UNSUPPORTED;
    if (opt->schedule < 0 || opt->schedule > 4) return QOQ_ERR_UNSUPPORTED;
    return QOQ_OK;
}

bool plan_for(int M, int N, int K, int group, const qoq_gemm_options *opt, qoq::GemmPlan *out) {
    const int sms = num_sms_current_device();
    if (sms <= 0) return false;
    *out = qoq::plan_gemm(M, N, K, group, sms, opt ? opt->kernel : 0, opt ? opt->tokens_per_tile : 0,
                          opt ? opt->num_ctas : 0, !(opt && (opt->flags & QOQ_PLAN_RULES)),
                          opt ? opt->schedule : 0);
    return true;
}

// A plan the kernels can run (path 0: a forced path that does not take this shape).
bool plan_valid(const qoq::GemmPlan &plan) { return plan.path >= 1 && plan.path <= 3; }

int gemm_common(const int8_t *Qx, const uint16_t *s_x, const int32_t *t_x, const void *packed,
                const uint16_t *s_w, int M, int N, int K, int group, uint16_t *O, int32_t *acc_out,
                void *ws, size_t ws_bytes, const qoq_gemm_options *opt, cudaStream_t stream) {
    const void *act = opt ? opt->act_operand : nullptr;
    if (act && !aligned(act, 16)) return QOQ_ERR_MISALIGNED;
    int st = check_gemm_shape(M, N, K, group);
    if (st != QOQ_OK) return st;
    st = check_options(opt);
    if (st != QOQ_OK) return st;
    if (!Qx || !packed || !ws) return QOQ_ERR_INVALID_ARG;
    if (group == 0 && !t_x) return QOQ_ERR_INVALID_ARG;
    if (!acc_out && (!O || !s_x || !s_w)) return QOQ_ERR_INVALID_ARG;
    if (!aligned(Qx, 16) || !aligned(packed, 16) || !aligned(ws, 16)) return QOQ_ERR_MISALIGNED;
    if ((s_x && !aligned(s_x, 2)) || (s_w && !aligned(s_w, 2)) || (O && !aligned(O, 16)) ||
        (t_x && !aligned(t_x, 4)) || (acc_out && !aligned(acc_out, 4)))
        return QOQ_ERR_MISALIGNED;
    st = check_current_device();
    if (st != QOQ_OK) return st;
    qoq::GemmPlan plan;
    if (!plan_for(M, N, K, group, opt, &plan)) return QOQ_ERR_CUDA;
    if (!plan_valid(plan)) return QOQ_ERR_UNSUPPORTED;
    if (plan.total * (plan.ctas + 1ll) >= (1ll << 32)) return QOQ_ERR_UNSUPPORTED;
    if (ws_bytes < plan.ws_bytes) return QOQ_ERR_WORKSPACE;
    qoq::GemmArgs a;
    a.Qx = Qx;
    a.s_x = s_x;
    a.t_x = t_x;
    a.packed = packed;
    a.s_w = s_w;
    a.M = M;
    a.N = N;
    a.K = K;
    a.group = group;
    a.act = act;
    a.O = O;
    a.acc_out = acc_out;
    a.ws = ws;
    a.debug_flags = opt ? opt->debug_flags : 0u;
    a.timeout_ns = (opt && opt->timeout_ns) ? opt->timeout_ns : kDefaultTimeoutNs;
    a.pdl = opt && (opt->flags & QOQ_LAUNCH_OVERLAP) != 0;
    return cuda_status(qoq::launch_gemm(a, plan, stream));
}

}  // namespace

extern "C" {

const char *qoq_status_string(int status) {
    switch (status) {
        case QOQ_OK: return "QOQ_OK";
        case QOQ_ERR_INVALID_ARG: return "QOQ_ERR_INVALID_ARG";
        case QOQ_ERR_UNSUPPORTED: return "QOQ_ERR_UNSUPPORTED";
        case QOQ_ERR_MISALIGNED: return "QOQ_ERR_MISALIGNED";
        case QOQ_ERR_WORKSPACE: return "QOQ_ERR_WORKSPACE";
        case QOQ_ERR_CUDA: return "QOQ_ERR_CUDA";
        case QOQ_ERR_TIMEOUT: return "QOQ_ERR_TIMEOUT";
        case QOQ_ERR_DEVICE: return "QOQ_ERR_DEVICE";
        default: return "QOQ_ERR_UNKNOWN";
    }
}

int qoq_version(void) { return static_cast<int>(qoq::kPackedVersion); }

int qoq_bounds_checked(void) {
#ifdef QOQ_DEBUG_BOUNDS
    return 1;
#else
    return 0;
#endif
}

int qoq_quantize_weights(const uint16_t *W, int N, int K, int group, uint8_t *q4, uint8_t *s_g,
                         uint8_t *z, uint16_t *s_w, qoq_stream_t stream) {
    if (N <= 0 || K <= 0) return QOQ_ERR_INVALID_ARG;
    if (group != 0 && group != 128) return QOQ_ERR_UNSUPPORTED;
    if (group == 128 && K % 128 != 0) return QOQ_ERR_UNSUPPORTED;
    if (!W || !q4 || !z || !s_w || (group && !s_g)) return QOQ_ERR_INVALID_ARG;
    if (!aligned(W, 2) || !aligned(s_w, 2)) return QOQ_ERR_MISALIGNED;
    return cuda_status(qoq::launch_quantize_weights(W, N, K, group, q4, s_g, z, s_w,
                                                    reinterpret_cast<cudaStream_t>(stream)));
}

size_t qoq_packed_weight_bytes(int N, int K, int group) {
    if (N <= 0 || K <= 0 || N % 128 || K % 128 || (group != 0 && group != 128)) return 0;
    return qoq::packed_bytes(N, K, group);
}

int qoq_pack_weights(const uint8_t *q4, const uint8_t *s_g, const uint8_t *z, int N, int K,
                     int group, void *packed, qoq_stream_t stream) {
    if (N <= 0 || K <= 0) return QOQ_ERR_INVALID_ARG;
    if (group != 0 && group != 128) return QOQ_ERR_UNSUPPORTED;
    if (N % 128 || K % 128 || N / 128 > 65535) return QOQ_ERR_UNSUPPORTED;
    if (!q4 || !z || !packed || (group && !s_g)) return QOQ_ERR_INVALID_ARG;
    if (!aligned(q4, 16) || !aligned(packed, 16)) return QOQ_ERR_MISALIGNED;
    return cuda_status(qoq::launch_pack(q4, s_g, z, N, K, group, packed,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

int qoq_unpack_weights(const void *packed, int N, int K, int group, uint8_t *q4, uint8_t *s_g,
                       uint8_t *z, qoq_stream_t stream) {
    if (N <= 0 || K <= 0) return QOQ_ERR_INVALID_ARG;
    if (group != 0 && group != 128) return QOQ_ERR_UNSUPPORTED;
    if (N % 128 || K % 128 || N / 128 > 65535) return QOQ_ERR_UNSUPPORTED;
    if (!q4 || !z || !packed || (group && !s_g)) return QOQ_ERR_INVALID_ARG;
    if (!aligned(q4, 16) || !aligned(packed, 16)) return QOQ_ERR_MISALIGNED;
    return cuda_status(qoq::launch_unpack(packed, N, K, group, q4, s_g, z,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

int qoq_quant_act(const uint16_t *X, int M, int K, int8_t *Qx, uint16_t *s_x, int32_t *t_x,
                  qoq_stream_t stream) {
    if (M <= 0 || K <= 0) return QOQ_ERR_INVALID_ARG;
    if (K % 8 != 0) return QOQ_ERR_UNSUPPORTED;
    if (!X || !Qx || !s_x) return QOQ_ERR_INVALID_ARG;
    if (!aligned(X, 16) || !aligned(Qx, 16) || !aligned(s_x, 2) || (t_x && !aligned(t_x, 4)))
        return QOQ_ERR_MISALIGNED;
    return cuda_status(
        qoq::launch_quant_act(X, M, K, Qx, s_x, t_x, 0, nullptr, false, reinterpret_cast<cudaStream_t>(stream)));
}

size_t qoq_act_operand_bytes(int M, int K, int kind) {
    if (M <= 0 || K <= 0 || K % 128 != 0 || (kind != 1 && kind != 2)) return 0;  // kind 3 reads Qx: none
    return qoq::act_operand_bytes(M, K, kind);
}

int qoq_quant_act_ex(const uint16_t *X, int M, int K, int8_t *Qx, uint16_t *s_x, int32_t *t_x,
                     int kind, void *act_operand, uint32_t flags, qoq_stream_t stream) {
    if (M <= 0 || K <= 0) return QOQ_ERR_INVALID_ARG;
    if (flags & ~QOQ_LAUNCH_OVERLAP) return QOQ_ERR_UNSUPPORTED;
    if (act_operand && kind != 1 && kind != 2 && kind != 3) return QOQ_ERR_INVALID_ARG;
    if (kind == 3) act_operand = nullptr;  // the CUDA-core path reads Qx itself
    if (K % 8 != 0 || (act_operand && K % 128 != 0)) return QOQ_ERR_UNSUPPORTED;
    if (!X || !Qx || !s_x) return QOQ_ERR_INVALID_ARG;
    if (!aligned(X, 16) || !aligned(Qx, 16) || !aligned(s_x, 2) || (t_x && !aligned(t_x, 4)) ||
        (act_operand && !aligned(act_operand, 16)))
        return QOQ_ERR_MISALIGNED;
    return cuda_status(
        qoq::launch_quant_act(X, M, K, Qx, s_x, t_x, act_operand ? kind : 0, act_operand,
                              (flags & QOQ_LAUNCH_OVERLAP) != 0, reinterpret_cast<cudaStream_t>(stream)));
}

int qoq_rmsnorm_quant_act(const uint16_t *X, const uint16_t *gamma, float eps, int M, int K, int8_t *Qx,
                          uint16_t *s_x, int32_t *t_x, int kind, void *act_operand, uint16_t *Y, uint32_t flags,
                          qoq_stream_t stream) {
    if (M <= 0 || K <= 0) return QOQ_ERR_INVALID_ARG;
    if (!(eps >= 0.0f) || eps > 3.0e38f) return QOQ_ERR_INVALID_ARG;  // rejects NaN and inf too
    if (flags & ~QOQ_LAUNCH_OVERLAP) return QOQ_ERR_UNSUPPORTED;
    if (act_operand && kind != 1 && kind != 2 && kind != 3) return QOQ_ERR_INVALID_ARG;
    if (kind == 3) act_operand = nullptr;  // the CUDA-core path reads Qx itself
    if (K % 8 != 0 || (act_operand && K % 128 != 0)) return QOQ_ERR_UNSUPPORTED;
    if (!X || !gamma || !Qx || !s_x) return QOQ_ERR_INVALID_ARG;
    if (!aligned(X, 16) || !aligned(gamma, 16) || !aligned(Qx, 16) || !aligned(s_x, 2) ||
        (t_x && !aligned(t_x, 4)) || (act_operand && !aligned(act_operand, 16)) || (Y && !aligned(Y, 16)))
        return QOQ_ERR_MISALIGNED;
    return cuda_status(qoq::launch_rmsnorm_quant(X, gamma, eps, Y, M, K, Qx, s_x, t_x, act_operand ? kind : 0,
                                                 act_operand, (flags & QOQ_LAUNCH_OVERLAP) != 0,
                                                 reinterpret_cast<cudaStream_t>(stream)));
}

int qoq_silu_mul_quant_act(const uint16_t *H, int M, int F, int8_t *Qx, uint16_t *s_x, int32_t *t_x, int kind,
                           void *act_operand, uint16_t *Y, uint32_t flags, qoq_stream_t stream) {
    if (M <= 0 || F <= 0) return QOQ_ERR_INVALID_ARG;
    if (flags & ~QOQ_LAUNCH_OVERLAP) return QOQ_ERR_UNSUPPORTED;
    if (act_operand && kind != 1 && kind != 2 && kind != 3) return QOQ_ERR_INVALID_ARG;
    if (kind == 3) act_operand = nullptr;  // the CUDA-core path reads Qx itself
    if (F % 8 != 0 || (act_operand && F % 128 != 0)) return QOQ_ERR_UNSUPPORTED;
    if (!H || !Qx || !s_x) return QOQ_ERR_INVALID_ARG;
    if (!aligned(H, 16) || !aligned(Qx, 16) || !aligned(s_x, 2) || (t_x && !aligned(t_x, 4)) ||
        (act_operand && !aligned(act_operand, 16)) || (Y && !aligned(Y, 16)))
        return QOQ_ERR_MISALIGNED;
    return cuda_status(qoq::launch_silu_mul_quant(H, Y, M, F, Qx, s_x, t_x, act_operand ? kind : 0, act_operand,
                                                  (flags & QOQ_LAUNCH_OVERLAP) != 0,
                                                  reinterpret_cast<cudaStream_t>(stream)));
}

size_t qoq_gemm_workspace_bytes_ex(int M, int N, int K, int group, const qoq_gemm_options *opt) {
    if (check_gemm_shape(M, N, K, group) != QOQ_OK || check_options(opt) != QOQ_OK) return 0;
    qoq::GemmPlan plan;
    if (!plan_for(M, N, K, group, opt, &plan) || !plan_valid(plan)) return 0;
    return plan.ws_bytes;
}

size_t qoq_gemm_workspace_bytes(int M, int N, int K, int group) {
    return qoq_gemm_workspace_bytes_ex(M, N, K, group, nullptr);
}

int qoq_gemm_path(int M, int N, int K, int group, const qoq_gemm_options *opt) {
    int st = check_gemm_shape(M, N, K, group);
    if (st != QOQ_OK) return -st;
    st = check_options(opt);
    if (st != QOQ_OK) return -st;
    qoq::GemmPlan plan;
    if (!plan_for(M, N, K, group, opt, &plan)) return -QOQ_ERR_CUDA;
    if (!plan_valid(plan)) return -QOQ_ERR_UNSUPPORTED;
    return plan.path;
}

int qoq_gemm_plan(int M, int N, int K, int group, int num_sms, const qoq_gemm_options *opt,
                  qoq_gemm_plan_info *out) {
    if (!out || num_sms <= 0) return QOQ_ERR_INVALID_ARG;
    int st = check_gemm_shape(M, N, K, group);
    if (st != QOQ_OK) return st;
    st = check_options(opt);
    if (st != QOQ_OK) return st;
    const qoq::GemmPlan plan = qoq::plan_gemm(M, N, K, group, num_sms, opt ? opt->kernel : 0,
                                              opt ? opt->tokens_per_tile : 0, opt ? opt->num_ctas : 0,
                                              !(opt && (opt->flags & QOQ_PLAN_RULES)), opt ? opt->schedule : 0);
    if (!plan_valid(plan)) return QOQ_ERR_UNSUPPORTED;
    out->path = plan.path;
    out->tokens_per_tile = plan.BT;
    out->num_ctas = plan.ctas;
    out->tiles = plan.tiles;
    out->k_stages = plan.total;
    out->workspace_bytes = plan.ws_bytes;
    return QOQ_OK;
}

int qoq_workspace_init(void *workspace, size_t bytes, qoq_stream_t stream) {
    if (!workspace || bytes == 0) return QOQ_ERR_INVALID_ARG;
    return cuda_status(cudaMemsetAsync(workspace, 0, bytes, reinterpret_cast<cudaStream_t>(stream)));
}

int qoq_w4a8_gemm(const int8_t *Qx, const uint16_t *s_x, const int32_t *t_x, const void *packed,
                  const uint16_t *s_w, int M, int N, int K, int group, uint16_t *O,
                  void *workspace, size_t ws_bytes, qoq_stream_t stream) {
    return gemm_common(Qx, s_x, t_x, packed, s_w, M, N, K, group, O, nullptr, workspace, ws_bytes,
                       nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int qoq_w4a8_gemm_i32(const int8_t *Qx, const int32_t *t_x, const void *packed, int M, int N,
                      int K, int group, int32_t *acc, void *workspace, size_t ws_bytes,
                      qoq_stream_t stream) {
    if (!acc) return QOQ_ERR_INVALID_ARG;
    return gemm_common(Qx, nullptr, t_x, packed, nullptr, M, N, K, group, nullptr, acc, workspace,
                       ws_bytes, nullptr, reinterpret_cast<cudaStream_t>(stream));
}

int qoq_w4a8_gemm_ex(const int8_t *Qx, const uint16_t *s_x, const int32_t *t_x,
                     const void *packed, const uint16_t *s_w, int M, int N, int K, int group,
                     uint16_t *O, void *workspace, size_t ws_bytes, const qoq_gemm_options *opt,
                     qoq_stream_t stream) {
    return gemm_common(Qx, s_x, t_x, packed, s_w, M, N, K, group, O, opt ? opt->acc_out : nullptr,
                       workspace, ws_bytes, opt, reinterpret_cast<cudaStream_t>(stream));
}

size_t qoq_kv4_page_bytes(int num_kv_heads) {
    if (num_kv_heads <= 0 || num_kv_heads > 1024) return 0;
    return static_cast<size_t>(num_kv_heads) * qoq::kKv4HeadChunkBytes;
}

int qoq_kv4_append(const uint16_t *K, const uint16_t *V, int num_tokens, int num_kv_heads, const int32_t *token_seq,
                   const int32_t *token_pos, const int32_t *page_table, int num_seqs, int max_pages, void *pages,
                   int num_pages, uint32_t *status, qoq_stream_t stream) {
    if (num_tokens <= 0 || num_kv_heads <= 0 || num_kv_heads > 1024 || num_seqs <= 0 || max_pages <= 0 ||
        num_pages <= 0)
        return QOQ_ERR_INVALID_ARG;
    if (!K || !V || !token_seq || !token_pos || !page_table || !pages) return QOQ_ERR_INVALID_ARG;
    if (!aligned(K, 16) || !aligned(V, 16) || !aligned(pages, 16) || !aligned(token_seq, 4) ||
        !aligned(token_pos, 4) || !aligned(page_table, 4) || (status && !aligned(status, 4)))
        return QOQ_ERR_MISALIGNED;
    int st = check_current_device();
    if (st != QOQ_OK) return st;
    return cuda_status(qoq::launch_kv4_append(K, V, num_tokens, num_kv_heads, token_seq, token_pos, page_table,
                                              num_seqs, max_pages, num_pages, pages, status,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
int check_kv4_attention_shape(int B, int num_q_heads, int num_kv_heads, int max_pages) {
    if (B <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_pages <= 0) return QOQ_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads != 0) return QOQ_ERR_UNSUPPORTED;
    const int G = num_q_heads / num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8) return QOQ_ERR_UNSUPPORTED;
    if (num_kv_heads > 65535 || B > 65535) return QOQ_ERR_UNSUPPORTED;
    return QOQ_OK;
}
}  // namespace

size_t qoq_kv4_attention_workspace_bytes(int B, int num_q_heads, int num_kv_heads, int max_pages) {
    if (check_kv4_attention_shape(B, num_q_heads, num_kv_heads, max_pages) != QOQ_OK) return 0;
    const int sms = num_sms_current_device();
    if (sms <= 0) return 0;
    return qoq::plan_kv4_attention(B, num_q_heads, num_kv_heads, max_pages, sms).ws_bytes;
}

int qoq_kv4_decode_attention(const uint16_t *Q, const void *pages, int num_pages, const int32_t *page_table,
                             const int32_t *seq_lens, int B, int num_q_heads, int num_kv_heads, int max_pages,
                             float softmax_scale, uint16_t *O, void *workspace, size_t ws_bytes,
                             qoq_stream_t stream) {
    int st = check_kv4_attention_shape(B, num_q_heads, num_kv_heads, max_pages);
    if (st != QOQ_OK) return st;
    if (num_pages <= 0 || !(softmax_scale > 0.0f) || softmax_scale > 3.0e38f) return QOQ_ERR_INVALID_ARG;
    if (!Q || !pages || !page_table || !seq_lens || !O || !workspace) return QOQ_ERR_INVALID_ARG;
    if (!aligned(Q, 16) || !aligned(O, 16) || !aligned(pages, 16) || !aligned(page_table, 4) ||
        !aligned(seq_lens, 4) || !aligned(workspace, 16))
        return QOQ_ERR_MISALIGNED;
    st = check_current_device();
    if (st != QOQ_OK) return st;
    const int sms = num_sms_current_device();
    if (sms <= 0) return QOQ_ERR_CUDA;
    const qoq::Kv4Plan plan = qoq::plan_kv4_attention(B, num_q_heads, num_kv_heads, max_pages, sms);
    if (ws_bytes < plan.ws_bytes) return QOQ_ERR_WORKSPACE;
    return cuda_status(qoq::launch_kv4_attention(Q, pages, page_table, seq_lens, B, num_q_heads, num_kv_heads,
                                                 max_pages, num_pages, softmax_scale, O, workspace, plan,
                                                 kDefaultTimeoutNs, reinterpret_cast<cudaStream_t>(stream)));
}

int qoq_workspace_status(void *workspace, uint32_t *host_status, qoq_stream_t stream) {
    if (!workspace || !host_status) return QOQ_ERR_INVALID_ARG;
    if (!aligned(workspace, 16)) return QOQ_ERR_MISALIGNED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(v), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return QOQ_ERR_CUDA;
    *host_status = v;
    if (v & 8u) return QOQ_ERR_DEVICE;  // bounds-check build: a skipped access, the cause of any expired wait
    if (v & 1u) return QOQ_ERR_TIMEOUT;
    if (v & 6u) return QOQ_ERR_DEVICE;
    return QOQ_OK;
}

}  // extern "C"
