// gdn_noalloc.cu -- chunked prefill that needs no caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they run a prefill:
// engines whose device memory is carved up once at start-up by their own pool and
// that have no hook to hand a kernel extra scratch, plugins that only ever see the
// input and output buffers their host passes them, and deployments that forbid any
// allocation after initialisation (cudaMalloc may also synchronise the device, which
// a latency-critical path cannot afford).  gdn_prefill_noalloc serves them: its
// scratch is a file-scope __device__ array of kScratchBytes that every GPU which loads
// this library holds until the process exits.  The caller still passes every input
// and output buffer.  Nothing here calls cudaMalloc, cudaFree or an allocating
// library routine.
#include <math.h>
#include <atomic>
#include <string.h>

#include "gdn_internal.cuh"

namespace {

constexpr size_t kScratchBytes = (size_t)64 << 20;     // 64 MiB per device
__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void *> g_scratch_addr[kMaxDevices];

// Device address of g_scratch on the current device.  In host code the array's name
// is only a host-side stand-in, so the address is asked for with that device current.
// Only a successful lookup is kept: a lookup that failed (made during a stream capture,
// or with an error left by earlier work) is tried again on the next call.
int scratch_for_current_device(void **addr) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return GDN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_UNSUPPORTED;
    void *a = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (a == nullptr) {
        if (cudaGetSymbolAddress(&a, g_scratch) != cudaSuccess || a == nullptr) return GDN_ERR_CUDA;
        g_scratch_addr[dev].store(a, std::memory_order_release);
    }
    *addr = a;
    return GDN_OK;
}

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

extern "C" int gdn_prefill_noalloc(const void *queries, const void *keys, const void *values,
                                   const float *decays, const float *beta,
                                   const float *initial_state, void *out, float *final_state,
                                   float *states, int B, int T, int HK, int HV, int Dk, int Dv,
                                   gdn_dtype dtype, float scale, int use_qk_l2norm,
                                   void *cuda_stream) {
    using namespace gdn;
    // the same argument rules as gdn_prefill
    if (B < 0 || T < 0 || HK <= 0 || HV <= 0 || HV % HK != 0) return GDN_ERR_INVALID_ARG;
    if (!(Dk == 32 || Dk == 64 || Dk == 128) || Dv != Dk) return GDN_ERR_UNSUPPORTED;
    if (dtype != GDN_BF16 && dtype != GDN_F32) return GDN_ERR_UNSUPPORTED;
    if (isnan(scale) || isinf(scale)) return GDN_ERR_INVALID_ARG;
    if (B > 65535 || HV > 65535 || (int64_t)B * T > INT32_MAX) return GDN_ERR_UNSUPPORTED;
    if ((int64_t)B * HV * kChainSlices > INT32_MAX) return GDN_ERR_UNSUPPORTED;   // chain numbers
    const int64_t T_total = (int64_t)B * T;
    if (B > 0 && !final_state) return GDN_ERR_INVALID_ARG;
    if (T_total > 0 && (!queries || !keys || !values || !decays || !beta || !out))
        return GDN_ERR_INVALID_ARG;
    const void *ptrs[] = {queries, keys, values, decays, beta, initial_state, out, final_state, states};
    for (const void *p : ptrs)
        if (p && ((uintptr_t)p & 15u)) return GDN_ERR_MISALIGNED;

    // scratch needed by the kernels this shape runs: status words, then one record
    // per (chunk, value head)
    const int mc = B * ((T + kChunk - 1) / kChunk);
    const bool tc = tc_supported(Dk, Dv, dtype);
    const size_t rec_bytes = tc ? tc_record_bytes() : record_floats(Dk, Dv) * sizeof(float);
    const size_t table = round256(sizeof(int32_t) * ((size_t)mc + B + 1));
    const size_t flag_bytes = chain_flag_bytes(B, HV) + ready_flag_bytes(mc, HV);
    const size_t need = kWsHeader + flag_bytes + table + (size_t)mc * HV * rec_bytes;
    if (need > kScratchBytes) return GDN_ERR_WORKSPACE;     // beyond the fixed maximum

    void *scratch = nullptr;
    int rc = scratch_for_current_device(&scratch);
    if (rc != GDN_OK) return rc;
    cudaStream_t st = (cudaStream_t)cuda_stream;
    // the array keeps the previous call's contents: start from clean status and flag words
    if (cudaMemsetAsync(scratch, 0, kWsHeader + flag_bytes, st) != cudaSuccess) return GDN_ERR_CUDA;
    if (B == 0) return GDN_OK;

    char *ws = (char *)scratch;
    PrefillParams p;
    memset(&p, 0, sizeof p);
    p.q = queries; p.k = keys; p.v = values; p.g = decays; p.beta = beta;
    p.s0 = initial_state; p.out = out; p.s_final = final_state; p.states = states;
    p.cu_seqlens = nullptr;
    p.N = B; p.T_seq = T; p.T_total = T_total;
    p.HK = HK; p.HV = HV; p.Dk = Dk; p.Dv = Dv;
    p.scale = scale > 0.f ? scale : 1.0f / sqrtf((float)Dk);
    p.l2norm = use_qk_l2norm ? 1 : 0;
    p.max_chunks = mc;
    p.status = (int32_t *)ws;
    p.chain_flags = (int32_t *)(ws + kWsHeader);
    p.ready = (int32_t *)(ws + kWsHeader + chain_flag_bytes(B, HV));
    p.chunk_seq = (int32_t *)(ws + kWsHeader + flag_bytes);
    p.chunk_first = p.chunk_seq + mc;
    p.rec = (float *)(ws + kWsHeader + flag_bytes + table);
    p.rec_floats = tc ? tc_record_bytes() / sizeof(float) : record_floats(Dk, Dv);
    cudaError_t e = tc ? launch_prefill_tc(p, st) : launch_prefill_generic(p, dtype, st);
    return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA;
}

extern "C" int gdn_prefill_noalloc_status(void *cuda_stream, int *status) {
    using namespace gdn;
    if (!status) return GDN_ERR_INVALID_ARG;
    void *scratch = nullptr;
    int rc = scratch_for_current_device(&scratch);
    if (rc != GDN_OK) return rc;
    int32_t v = 0;
    cudaStream_t st = (cudaStream_t)cuda_stream;
    if (cudaMemcpyAsync(&v, scratch, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess) return GDN_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return GDN_ERR_CUDA;
    *status = v;
    return GDN_OK;
}
