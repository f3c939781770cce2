// ssd_api.cu -- the C ABI declared in include/ssd.h: argument validation,
// plan choice, workspace layout and launches.  Everything here runs on the
// host; nothing allocates device memory or synchronises a stream except
// ssd_check_device_error.  ssd_fwd_host creates, once per device, two copy
// streams and four events for its pipeline.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "ssd_fused.cuh"
#include "ssd_internal.cuh"

namespace {

thread_local char g_detail[512] = "";

ssd_status fail(ssd_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_detail, sizeof(g_detail), fmt, ap);
    va_end(ap);
    return st;
}

ssd_status ok() {
    g_detail[0] = '\0';
    return SSD_OK;
}

ssd_status cuda_fail(cudaError_t e, const char *where) {
    return fail(SSD_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

constexpr size_t kAlign = 256;
size_t align_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

size_t io_size(int32_t dt) { return dt == SSD_F32 ? 4 : 2; }

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Shape and dtype checks shared by every entry point (pointers excluded).
ssd_status check_shape(const ssd_fwd_args *a) {
    if (!a) return fail(SSD_ERR_INVALID_ARG, "args is NULL");
    if (a->B <= 0 || a->L <= 0 || a->H <= 0 || a->P <= 0 || a->N <= 0 || a->G <= 0 || a->chunk <= 0)
        return fail(SSD_ERR_INVALID_ARG, "every dim must be > 0 (B=%lld L=%lld H=%lld P=%lld N=%lld G=%lld chunk=%lld)",
                    (long long)a->B, (long long)a->L, (long long)a->H, (long long)a->P,
                    (long long)a->N, (long long)a->G, (long long)a->chunk);
    if (a->H % a->G != 0)
        return fail(SSD_ERR_INVALID_ARG, "H (%lld) must be a multiple of G (%lld)", (long long)a->H,
                    (long long)a->G);
    if (a->chunk < 16 || a->chunk > 256 || a->chunk % 16 != 0)
        return fail(SSD_ERR_UNSUPPORTED, "chunk must be a multiple of 16 in [16, 256] (got %lld)",
                    (long long)a->chunk);
    if (a->P % 16 != 0 || a->P > 128 || a->N % 16 != 0 || a->N > 128)
        return fail(SSD_ERR_UNSUPPORTED, "P and N must be multiples of 16 up to 128 (P=%lld N=%lld)",
                    (long long)a->P, (long long)a->N);
    const int64_t nchunks = (a->L + a->chunk - 1) / a->chunk;
    if (a->B > 65535 || nchunks > 65535 || a->B * a->H > 0x7fffffffLL || a->L > 0x7fffffffLL)
        return fail(SSD_ERR_UNSUPPORTED, "B <= 65535, ceil(L/chunk) <= 65535 and B*H, L < 2^31 required");
    for (int32_t d : {a->x_dtype, a->bc_dtype, a->y_dtype})
        if (d != SSD_F32 && d != SSD_F16 && d != SSD_BF16)
            return fail(SSD_ERR_INVALID_ARG, "unknown dtype code %d", d);
    if (a->bc_dtype != a->x_dtype || a->y_dtype != a->x_dtype)
        return fail(SSD_ERR_UNSUPPORTED, "x, B, C and y must share one dtype");
    if (a->z && a->z_dtype != a->x_dtype)
        return fail(SSD_ERR_UNSUPPORTED, "z must have the dtype of x");
    if (a->ops != SSD_OPS_F32 && a->ops != SSD_OPS_F16 && a->ops != SSD_OPS_BF16)
        return fail(SSD_ERR_INVALID_ARG, "unknown operand mode %d", a->ops);
    if (a->plan != SSD_PLAN_AUTO && a->plan != SSD_PLAN_CHUNKED && a->plan != SSD_PLAN_FUSED)
        return fail(SSD_ERR_INVALID_ARG, "unknown plan %d", a->plan);
    if (!(a->dt_min <= a->dt_max) || isnan(a->dt_min) || isnan(a->dt_max))
        return fail(SSD_ERR_INVALID_ARG, "dt_limit must satisfy dt_min <= dt_max");
    if (a->conv_width < 0 || a->conv_width > 4)
        return fail(SSD_ERR_UNSUPPORTED, "conv_width must be 0 (no convolution) or 1..4 (got %d)", a->conv_width);
    return SSD_OK;
}

ssd_status check_pointers(const ssd_fwd_args *a, bool need_y) {
    if (!a->x || !a->dt || !a->A || !a->Bm || !a->Cm)
        return fail(SSD_ERR_INVALID_ARG, "x, dt, A, B and C are required");
    if (need_y && !a->y) return fail(SSD_ERR_INVALID_ARG, "y is required");
    if (a->initial_state && !aligned(a->initial_state, 16))
        return fail(SSD_ERR_INVALID_ARG, "initial_state must be 16-byte aligned");
    if (a->final_state && !aligned(a->final_state, 16))
        return fail(SSD_ERR_INVALID_ARG, "final_state must be 16-byte aligned");
    if (a->norm_weight && !a->z) return fail(SSD_ERR_INVALID_ARG, "the gated RMSNorm (norm_weight) needs z");
    if (a->norm_weight && !(a->norm_eps >= 0.f && a->norm_eps < INFINITY))
        return fail(SSD_ERR_INVALID_ARG, "norm_eps must be finite and >= 0");
    if (a->conv_width > 0) {
        if (!a->conv_x_weight || !a->conv_b_weight || !a->conv_c_weight)
            return fail(SSD_ERR_INVALID_ARG, "the conv1d (conv_width > 0) needs conv_x_weight, conv_b_weight and "
                                             "conv_c_weight");
        for (const void *ptr : {a->x, a->Bm, a->Cm})
            if (!aligned(ptr, 16)) return fail(SSD_ERR_UNSUPPORTED, "the conv1d needs 16-byte aligned x, B and C");
    }
    return SSD_OK;
}

// Entry points that take no convolution in front of the SSD.
ssd_status reject_conv(const ssd_fwd_args *a, const char *entry) {
    if (a && a->conv_width != 0) return fail(SSD_ERR_UNSUPPORTED, "%s does not take the conv1d (conv_width)", entry);
    return SSD_OK;
}

ssd::Params make_params(const ssd_fwd_args *a) {
    ssd::Params p;
    p.B = (int)a->B; p.L = (int)a->L; p.H = (int)a->H; p.P = (int)a->P; p.N = (int)a->N;
    p.G = (int)a->G; p.Q = (int)a->chunk;
    p.nchunks = (int)((a->L + a->chunk - 1) / a->chunk);
    p.hpg = (int)(a->H / a->G);
    p.x = a->x; p.dt = a->dt; p.A = a->A; p.Bm = a->Bm; p.Cm = a->Cm; p.D = a->D; p.z = a->z;
    p.dt_bias = a->dt_bias; p.h0 = a->initial_state; p.y = a->y; p.final_state = a->final_state;
    p.dt_softplus = a->dt_softplus ? 1 : 0;
    p.has_limit = !(a->dt_min == 0.f && isinf(a->dt_max) && a->dt_max > 0.f);
    p.dt_min = a->dt_min; p.dt_max = a->dt_max;
    return p;
}

struct ChunkedLayout {
    size_t err_off, dtp_off, cs_off, states_off, total;
};

ChunkedLayout chunked_layout(const ssd_fwd_args *a) {
    const size_t nchunks = (size_t)((a->L + a->chunk - 1) / a->chunk);
    const size_t vec = (size_t)a->B * a->H * nchunks * a->chunk * sizeof(float);
    const size_t st = (size_t)a->B * nchunks * a->H * a->P * a->N * sizeof(float);
    ChunkedLayout l;
    l.err_off = 0;
    l.dtp_off = kAlign;
    l.cs_off = l.dtp_off + align_up(vec);
    l.states_off = l.cs_off + align_up(vec);
    l.total = l.states_off + align_up(st);
    return l;
}

int32_t resolve_plan(const ssd_fwd_args *a) {
    if (a->plan != SSD_PLAN_AUTO) return a->plan;
    if (ssd::fused_supported(a) && ssd::fused_preferred(a)) return SSD_PLAN_FUSED;
    return SSD_PLAN_CHUNKED;
}

size_t plan_workspace(const ssd_fwd_args *a, int32_t plan) {
    if (plan == SSD_PLAN_FUSED) return ssd::fused_workspace_size(a);
    return chunked_layout(a).total;
}

// The causal conv1d in front of the SSD runs inside the fused kernel (N = 64);
// otherwise x, B and C are convolved into the workspace, after the plan's own
// part, by three launches of the token-major conv kernel.
bool conv_in_kernel(const ssd_fwd_args *a, int32_t plan) {
    return a->conv_width > 0 && plan == SSD_PLAN_FUSED && ssd::fused_conv_supported(a);
}

struct ConvLayout {
    size_t x, b, c, total;
};

ConvLayout conv_layout(const ssd_fwd_args *a, int32_t plan) {
    const size_t io = io_size(a->x_dtype);
    ConvLayout l;
    l.x = align_up(plan_workspace(a, plan));
    l.b = l.x + align_up((size_t)a->B * a->L * a->H * a->P * io);
    l.c = l.b + align_up((size_t)a->B * a->L * a->G * a->N * io);
    l.total = l.c + align_up((size_t)a->B * a->L * a->G * a->N * io);
    return l;
}

size_t workspace_for(const ssd_fwd_args *a, int32_t plan) {
    if (a->conv_width > 0 && !conv_in_kernel(a, plan)) return conv_layout(a, plan).total;
    return plan_workspace(a, plan);
}

// Steps 2 and 4 run on the tensor cores when the operands are fp16 / bf16 and
// the shape fits those kernels, else on the fp32 CUDA-core kernels.
bool tc_ok(const ssd_fwd_args *a) {
    for (const void *ptr : {static_cast<const void *>(a->x), static_cast<const void *>(a->Bm),
                            static_cast<const void *>(a->Cm)})
        if (reinterpret_cast<uintptr_t>(ptr) % 16 != 0) return false;
    return true;
}

cudaError_t launch_state_step(const ssd_fwd_args *a, const ssd::Params &p, const float *dtp, const float *cs,
                              float *states, unsigned int *err, cudaStream_t s) {
    if (ssd::chunk_tc_state_supported(p, a->ops) && tc_ok(a))
        return ssd::launch_chunk_state_tc(p, a->x_dtype, a->ops, dtp, cs, states, err, s);
    return ssd::launch_chunk_state(p, a->x_dtype, dtp, cs, states, s);
}

cudaError_t launch_scan_step(const ssd_fwd_args *a, const ssd::Params &p, const float *dtp, const float *cs,
                             const float *states, unsigned int *err, cudaStream_t s) {
    if (ssd::chunk_tc_scan_supported(p, a->ops) && tc_ok(a))
        return ssd::launch_chunk_scan_tc(p, a->x_dtype, a->ops, dtp, cs, states, err, s);
    return ssd::launch_chunk_scan(p, a->x_dtype, dtp, cs, states, s);
}

ssd_status run_chunked(const ssd_fwd_args *a, cudaStream_t s) {
    const ChunkedLayout l = chunked_layout(a);
    char *ws = static_cast<char *>(a->workspace);
    float *dtp = reinterpret_cast<float *>(ws + l.dtp_off);
    float *cs = reinterpret_cast<float *>(ws + l.cs_off);
    float *states = reinterpret_cast<float *>(ws + l.states_off);
    const ssd::Params p = make_params(a);
    // the chunked plan has no device-side waits; its error word is cleared so
    // that ssd_check_device_error reads "no error" after it
    cudaError_t e = cudaMemsetAsync(ws + l.err_off, 0, kAlign, s);
    if (e != cudaSuccess) return cuda_fail(e, "clearing the error word");
    if ((e = ssd::launch_chunk_cumsum(p, dtp, cs, s)) != cudaSuccess) return cuda_fail(e, "chunk_cumsum");
    unsigned int *err = reinterpret_cast<unsigned int *>(ws + l.err_off);
    if ((e = launch_state_step(a, p, dtp, cs, states, err, s)) != cudaSuccess) return cuda_fail(e, "chunk_state");
    if ((e = ssd::launch_state_passing(p, cs, states, s)) != cudaSuccess) return cuda_fail(e, "state_passing");
    if ((e = launch_scan_step(a, p, dtp, cs, states, err, s)) != cudaSuccess) return cuda_fail(e, "chunk_scan");
    return ok();
}

// The gated RMSNorm runs inside the fused kernel when it can; otherwise the
// forward runs without its z gate and a second kernel normalises y in place
// over `rows` tokens (the gate included).
bool norm_in_kernel(const ssd_fwd_args *a, int32_t plan) {
    return a->norm_weight && plan == SSD_PLAN_FUSED && ssd::fused_norm_supported(a) && a->conv_width == 0;
}

ssd_fwd_args without_norm(const ssd_fwd_args *a) {
    ssd_fwd_args o = *a;
    o.z = nullptr;
    o.norm_weight = nullptr;
    return o;
}

ssd_status norm_after(const ssd_fwd_args *a, int64_t rows, cudaStream_t s) {
    cudaError_t e = ssd::launch_gated_rmsnorm(rows, (int)(a->H * a->P), (int)a->G, a->norm_eps, a->x_dtype, a->y,
                                              a->z, a->norm_weight, a->y, s);
    if (e != cudaSuccess) return cuda_fail(e, "gated_rmsnorm");
    return ok();
}

// Packed variable-length input: checks of the offsets, the longest sequence.
ssd_status check_varlen(const ssd_fwd_args *a, const int64_t *cu, int64_t nseq, int64_t *max_len) {
    ssd_status st = check_shape(a);
    if (st != SSD_OK) return st;
    if (a->B != 1) return fail(SSD_ERR_INVALID_ARG, "packed sequences need B = 1 (got %lld)", (long long)a->B);
    if (!cu || nseq < 1) return fail(SSD_ERR_INVALID_ARG, "cu_seqlens and nseq >= 1 are required");
    if (nseq > 0x7fffffffLL / 64) return fail(SSD_ERR_UNSUPPORTED, "too many sequences");
    if (cu[0] != 0) return fail(SSD_ERR_INVALID_ARG, "cu_seqlens[0] must be 0");
    int64_t mx = 0;
    for (int64_t s = 0; s < nseq; ++s) {
        if (cu[s + 1] < cu[s])
            return fail(SSD_ERR_INVALID_ARG, "cu_seqlens must not decrease (entry %lld)", (long long)(s + 1));
        if (cu[s + 1] - cu[s] > mx) mx = cu[s + 1] - cu[s];
    }
    if (cu[nseq] != a->L)
        return fail(SSD_ERR_INVALID_ARG, "cu_seqlens[nseq] (%lld) must equal L (%lld)", (long long)cu[nseq],
                    (long long)a->L);
    *max_len = mx;
    return SSD_OK;
}

bool varlen_fused(const ssd_fwd_args *a, int64_t nseq) {
    if (a->plan == SSD_PLAN_CHUNKED || !ssd::fused_varlen_supported(a)) return false;
    // the host builds a schedule over the units: keep it small
    return (int64_t)nseq * a->G * ((a->H / a->G) / 2) <= (1LL << 24);
}

// one sequence's call of the chunked plan: B = 1 views into the packed tensors
ssd_fwd_args sequence_args(const ssd_fwd_args *a, const int64_t *cu, int64_t s) {
    ssd_fwd_args o = *a;
    const int64_t t0 = cu[s];
    o.B = 1;
    o.L = cu[s + 1] - cu[s];
    const size_t io = io_size(a->x_dtype);
    auto adv = [](const void *ptr, size_t bytes) -> const char * {
        return ptr ? static_cast<const char *>(ptr) + bytes : nullptr;
    };
    o.x = adv(a->x, (size_t)t0 * a->H * a->P * io);
    o.z = adv(a->z, (size_t)t0 * a->H * a->P * io);
    o.y = const_cast<char *>(adv(a->y, (size_t)t0 * a->H * a->P * io));
    o.dt = reinterpret_cast<const float *>(adv(a->dt, (size_t)t0 * a->H * 4));
    o.Bm = adv(a->Bm, (size_t)t0 * a->G * a->N * io);
    o.Cm = adv(a->Cm, (size_t)t0 * a->G * a->N * io);
    const size_t st = (size_t)s * a->H * a->P * a->N * 4;
    o.initial_state = reinterpret_cast<const float *>(adv(a->initial_state, st));
    o.final_state = reinterpret_cast<float *>(const_cast<char *>(adv(a->final_state, st)));
    return o;
}

size_t varlen_workspace(const ssd_fwd_args *a, int64_t nseq, int64_t max_len) {
    if (varlen_fused(a, nseq)) return ssd::fused_varlen_workspace_size(a, nseq);
    ssd_fwd_args o = *a;
    o.B = 1;
    o.L = max_len > 0 ? max_len : 1;
    return chunked_layout(&o).total;
}

struct BwdLayout {
    size_t dtp, cs, states, adj, dyp, ypre, dBh, dCh, partA, partD, partBias, total;
};

BwdLayout bwd_layout(const ssd_fwd_args *a) {
    const size_t c = (size_t)((a->L + a->chunk - 1) / a->chunk);
    const size_t vec = (size_t)a->B * a->H * c * a->chunk * 4;
    const size_t st = (size_t)a->B * c * a->H * a->P * a->N * 4;
    const size_t tok = (size_t)a->B * a->L * a->H * a->P;
    const size_t tokn = (size_t)a->B * a->L * a->H * a->N * 4;
    const size_t part = (size_t)a->B * c * a->H * 4;
    BwdLayout l;
    size_t o = kAlign;  // the error word (unused by the backward; kept for the forward steps)
    l.dtp = o; o += align_up(vec);
    l.cs = o; o += align_up(vec);
    l.states = o; o += align_up(st);
    l.adj = o; o += align_up(st);
    l.dyp = o; o += align_up(tok * 4);
    l.ypre = o; o += a->z ? align_up(tok * io_size(a->x_dtype)) : 0;
    l.dBh = o; o += align_up(tokn);
    l.dCh = o; o += align_up(tokn);
    l.partA = o; o += align_up(part);
    l.partD = o; o += align_up(part);
    l.partBias = o; o += align_up(part);
    l.total = o;
    return l;
}

ssd_status check_bwd(const ssd_bwd_args *b) {
    if (!b) return fail(SSD_ERR_INVALID_ARG, "args is NULL");
    const ssd_fwd_args *a = &b->fwd;
    ssd_status st = check_shape(a);
    if (st != SSD_OK) return st;
    if (a->norm_weight) return fail(SSD_ERR_UNSUPPORTED, "the backward does not take the gated RMSNorm");
    if ((st = reject_conv(a, "ssd_bwd")) != SSD_OK) return st;
    if (a->chunk > 64 || a->P > 64 || a->N > 64)
        return fail(SSD_ERR_UNSUPPORTED, "the backward needs chunk, P, N <= 64 (chunk=%lld P=%lld N=%lld)",
                    (long long)a->chunk, (long long)a->P, (long long)a->N);
    if ((st = check_pointers(a, false)) != SSD_OK) return st;
    if (!b->dy || !b->dx || !b->ddt || !b->dA || !b->dB || !b->dC)
        return fail(SSD_ERR_INVALID_ARG, "dy, dx, ddt, dA, dB and dC are required");
    if (a->D && !b->dD) return fail(SSD_ERR_INVALID_ARG, "dD is required when D is given");
    if (a->z && !b->dz) return fail(SSD_ERR_INVALID_ARG, "dz is required when z is given");
    if (a->dt_bias && !b->ddt_bias) return fail(SSD_ERR_INVALID_ARG, "ddt_bias is required when dt_bias is given");
    if ((b->dfinal && !aligned(b->dfinal, 16)) || (b->dh0 && !aligned(b->dh0, 16)))
        return fail(SSD_ERR_INVALID_ARG, "dfinal and dh0 must be 16-byte aligned");
    return SSD_OK;
}

}  // namespace

ssd_status ssd::report_error(ssd_status st, const char *msg) { return fail(st, "%s", msg); }

extern "C" {

int32_t ssd_abi_version(void) { return SSD_ABI_VERSION; }

const char *ssd_status_string(ssd_status st) {
    switch (st) {
        case SSD_OK: return "ok";
        case SSD_ERR_INVALID_ARG: return "invalid argument";
        case SSD_ERR_UNSUPPORTED: return "unsupported configuration";
        case SSD_ERR_WORKSPACE: return "workspace missing or too small";
        case SSD_ERR_CUDA: return "CUDA error";
        case SSD_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

const char *ssd_last_error_detail(void) { return g_detail; }

ssd_status ssd_fwd_resolve_plan(const ssd_fwd_args *a, int32_t *plan) {
    ssd_status st = check_shape(a);
    if (st != SSD_OK) return st;
    if (!plan) return fail(SSD_ERR_INVALID_ARG, "plan is NULL");
    const int32_t pl = resolve_plan(a);
    if (pl == SSD_PLAN_FUSED && !ssd::fused_supported(a))
        return fail(SSD_ERR_UNSUPPORTED, "the fused plan does not support this shape: %s",
                    ssd::fused_unsupported_reason(a));
    *plan = pl;
    return ok();
}

ssd_status ssd_fwd_workspace_size(const ssd_fwd_args *a, size_t *bytes) {
    int32_t plan = 0;
    ssd_status st = ssd_fwd_resolve_plan(a, &plan);
    if (st != SSD_OK) return st;
    if (!bytes) return fail(SSD_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = workspace_for(a, plan);
    return ok();
}

ssd_status ssd_fwd_describe(const ssd_fwd_args *a, char *out, size_t cap) {
    int32_t plan = 0;
    ssd_status st = ssd_fwd_resolve_plan(a, &plan);
    if (st != SSD_OK) return st;
    if (!out || cap == 0) return fail(SSD_ERR_INVALID_ARG, "out buffer required");
    const char *norm = a->norm_weight && !norm_in_kernel(a, plan) ? ",gated_rmsnorm" : "";
    const char *conv = a->conv_width > 0 && !conv_in_kernel(a, plan)
                           ? "conv_tokens_kernel,conv_tokens_kernel,conv_tokens_kernel,"
                           : "";
    if (plan == SSD_PLAN_FUSED) {
        const bool seg = ssd::fused_segments(a) > 1;
        snprintf(out, cap, "%s%sssd_fused_kernel%s", conv, seg ? "segment_state_kernel,segment_fold_kernel," : "",
                 norm);
        return ok();
    }
    const ssd::Params p = make_params(a);
    const bool tc_state = ssd::chunk_tc_state_supported(p, a->ops) && tc_ok(a);
    const bool tc_scan = ssd::chunk_tc_scan_supported(p, a->ops) && tc_ok(a);
    snprintf(out, cap, "%schunk_cumsum,%s,state_passing,%s%s", conv, tc_state ? "chunk_state_tc" : "chunk_state",
             tc_scan ? "chunk_scan_tc" : "chunk_scan", norm);
    return ok();
}

ssd_status ssd_fwd(const ssd_fwd_args *a, void *stream) {
    int32_t plan = 0;
    ssd_status st = ssd_fwd_resolve_plan(a, &plan);
    if (st != SSD_OK) return st;
    if ((st = check_pointers(a, true)) != SSD_OK) return st;
    const size_t need = workspace_for(a, plan);
    if (!a->workspace || a->workspace_bytes < need)
        return fail(SSD_ERR_WORKSPACE, "workspace of %zu bytes required (%zu given)", need,
                    a->workspace ? a->workspace_bytes : (size_t)0);
    if (!aligned(a->workspace, kAlign)) return fail(SSD_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (a->conv_width > 0 && !conv_in_kernel(a, plan)) {  // convolve x, B, C into the workspace, then the SSD
        const ConvLayout cl = conv_layout(a, plan);
        char *ws = static_cast<char *>(a->workspace);
        const int B = (int)a->B, L = (int)a->L, W = a->conv_width;
        cudaError_t e;
        if ((e = ssd::launch_conv_tokens(B, L, (int)(a->H * a->P), W, a->x_dtype, a->x, a->conv_x_weight,
                                         a->conv_x_bias, 1, ws + cl.x, s)) != cudaSuccess ||
            (e = ssd::launch_conv_tokens(B, L, (int)(a->G * a->N), W, a->x_dtype, a->Bm, a->conv_b_weight,
                                         a->conv_b_bias, 1, ws + cl.b, s)) != cudaSuccess ||
            (e = ssd::launch_conv_tokens(B, L, (int)(a->G * a->N), W, a->x_dtype, a->Cm, a->conv_c_weight,
                                         a->conv_c_bias, 1, ws + cl.c, s)) != cudaSuccess)
            return cuda_fail(e, "conv1d");
        ssd_fwd_args o = *a;
        o.x = ws + cl.x;
        o.Bm = ws + cl.b;
        o.Cm = ws + cl.c;
        o.conv_width = 0;
        return ssd_fwd(&o, stream);
    }
    if (a->norm_weight && !norm_in_kernel(a, plan)) {  // the forward without its gate, then the norm
        const ssd_fwd_args o = without_norm(a);
        if (plan == SSD_PLAN_FUSED) {
            cudaError_t e = ssd::run_fused(&o, s);
            if (e != cudaSuccess) return cuda_fail(e, "fused kernel");
        } else if ((st = run_chunked(&o, s)) != SSD_OK) {
            return st;
        }
        return norm_after(a, a->B * a->L, s);
    }
    if (plan == SSD_PLAN_FUSED) {
        cudaError_t e = ssd::run_fused(a, s);
        if (e != cudaSuccess) return cuda_fail(e, "fused kernel");
        return ok();
    }
    return run_chunked(a, s);
}

ssd_status ssd_fwd_varlen_workspace_size(const ssd_fwd_args *a, const int64_t *cu, int64_t nseq, size_t *bytes) {
    int64_t mx = 0;
    ssd_status st = reject_conv(a, "ssd_fwd_varlen");
    if (st != SSD_OK) return st;
    st = check_varlen(a, cu, nseq, &mx);
    if (st != SSD_OK) return st;
    if (!bytes) return fail(SSD_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = varlen_workspace(a, nseq, mx);
    return ok();
}

ssd_status ssd_fwd_varlen(const ssd_fwd_args *a, const int64_t *cu, int64_t nseq, void *stream) {
    int64_t mx = 0;
    ssd_status st = reject_conv(a, "ssd_fwd_varlen");
    if (st != SSD_OK) return st;
    st = check_varlen(a, cu, nseq, &mx);
    if (st != SSD_OK) return st;
    if (a->norm_weight) {  // the packed forward without its gate, then the norm over every token
        if ((st = check_pointers(a, true)) != SSD_OK) return st;
        const ssd_fwd_args o = without_norm(a);
        if ((st = ssd_fwd_varlen(&o, cu, nseq, stream)) != SSD_OK) return st;
        return norm_after(a, a->L, static_cast<cudaStream_t>(stream));
    }
    if (a->plan == SSD_PLAN_FUSED && !varlen_fused(a, nseq))
        return fail(SSD_ERR_UNSUPPORTED, "the fused plan does not support this shape: %s",
                    ssd::fused_unsupported_reason(a)  ? ssd::fused_unsupported_reason(a)
                    : !ssd::fused_varlen_supported(a) ? "packed sequences take it at N = 64 only"
                                                      : "too many units");
    if ((st = check_pointers(a, true)) != SSD_OK) return st;
    const size_t need = varlen_workspace(a, nseq, mx);
    if (!a->workspace || a->workspace_bytes < need)
        return fail(SSD_ERR_WORKSPACE, "workspace of %zu bytes required (%zu given)", need,
                    a->workspace ? a->workspace_bytes : (size_t)0);
    if (!aligned(a->workspace, kAlign)) return fail(SSD_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (varlen_fused(a, nseq)) {
        cudaError_t e = ssd::run_fused_varlen(a, cu, (int)nseq, s);
        if (e != cudaSuccess) return cuda_fail(e, "fused kernel");
        return ok();
    }
    for (int64_t q = 0; q < nseq; ++q) {
        const ssd_fwd_args o = sequence_args(a, cu, q);
        if (o.L == 0) {  // no tokens: the final state is the initial state
            if (!o.final_state) continue;
            const size_t bytes = (size_t)a->H * a->P * a->N * 4;
            cudaError_t e = o.initial_state
                                ? cudaMemcpyAsync(o.final_state, o.initial_state, bytes, cudaMemcpyDeviceToDevice, s)
                                : cudaMemsetAsync(o.final_state, 0, bytes, s);
            if (e != cudaSuccess) return cuda_fail(e, "empty sequence");
            continue;
        }
        if ((st = run_chunked(&o, s)) != SSD_OK) return st;
    }
    return ok();
}

ssd_status ssd_bwd_workspace_size(const ssd_bwd_args *b, size_t *bytes) {
    ssd_status st = check_bwd(b);
    if (st != SSD_OK) return st;
    if (!bytes) return fail(SSD_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = bwd_layout(&b->fwd).total;
    return ok();
}

ssd_status ssd_bwd(const ssd_bwd_args *b, void *stream) {
    ssd_status st = check_bwd(b);
    if (st != SSD_OK) return st;
    const ssd_fwd_args *a = &b->fwd;
    const BwdLayout l = bwd_layout(a);
    if (!b->workspace || b->workspace_bytes < l.total)
        return fail(SSD_ERR_WORKSPACE, "workspace of %zu bytes required (%zu given)", l.total,
                    b->workspace ? b->workspace_bytes : (size_t)0);
    if (!aligned(b->workspace, kAlign)) return fail(SSD_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(b->workspace);
    ssd::Params p = make_params(a);
    p.y = nullptr;
    p.final_state = nullptr;
    float *dtp = reinterpret_cast<float *>(ws + l.dtp), *cs = reinterpret_cast<float *>(ws + l.cs);
    float *states = reinterpret_cast<float *>(ws + l.states);
    // the forward's steps 1-3 (fp32 kernels): states entering every chunk
    cudaError_t e;
    if ((e = ssd::launch_chunk_cumsum(p, dtp, cs, s)) != cudaSuccess) return cuda_fail(e, "chunk_cumsum");
    if ((e = ssd::launch_chunk_state(p, a->x_dtype, dtp, cs, states, s)) != cudaSuccess)
        return cuda_fail(e, "chunk_state");
    if ((e = ssd::launch_state_passing(p, cs, states, s)) != cudaSuccess) return cuda_fail(e, "state_passing");
    void *ypre = nullptr;
    if (a->z) {  // y before the gate, for dz
        ypre = ws + l.ypre;
        ssd::Params q = p;
        q.z = nullptr;
        q.y = ypre;
        if ((e = ssd::launch_chunk_scan(q, a->x_dtype, dtp, cs, states, s)) != cudaSuccess)
            return cuda_fail(e, "chunk_scan");
    }
    ssd::BwdBuffers w;
    w.dtp = dtp; w.cs = cs; w.states = states;
    w.adj = reinterpret_cast<float *>(ws + l.adj);
    w.dy = b->dy; w.ypre = ypre;
    w.dyp = reinterpret_cast<float *>(ws + l.dyp);
    w.dfinal = b->dfinal;
    w.dx = b->dx; w.dz = b->dz; w.dB = b->dB; w.dC = b->dC;
    w.ddt = b->ddt; w.dA = b->dA; w.dD = b->dD; w.dbias = b->ddt_bias; w.dh0 = b->dh0;
    w.dBh = reinterpret_cast<float *>(ws + l.dBh);
    w.dCh = reinterpret_cast<float *>(ws + l.dCh);
    w.partA = reinterpret_cast<float *>(ws + l.partA);
    w.partD = reinterpret_cast<float *>(ws + l.partD);
    w.partBias = reinterpret_cast<float *>(ws + l.partBias);
    if ((e = ssd::launch_bwd(p, a->x_dtype, w, s)) != cudaSuccess) return cuda_fail(e, "backward");
    return ok();
}

ssd_status ssd_causal_conv1d_tokens(int64_t B, int64_t S, int64_t C, int64_t W, int32_t dtype, const void *x,
                                    const float *w, const float *bias, int32_t silu, void *out, void *stream) {
    if (B <= 0 || S <= 0 || C <= 0 || W <= 0)
        return fail(SSD_ERR_INVALID_ARG, "B, S, C, W must be > 0 (B=%lld S=%lld C=%lld W=%lld)", (long long)B,
                    (long long)S, (long long)C, (long long)W);
    if (W > 4) return fail(SSD_ERR_UNSUPPORTED, "W must be <= 4 (got %lld)", (long long)W);
    if (C % 4 != 0) return fail(SSD_ERR_UNSUPPORTED, "C must be a multiple of 4 (got %lld)", (long long)C);
    if (B > 65535 || (S + 15) / 16 > 65535 || C > 0x7fffffffLL || B * S * C > 0x7fffffffffffLL)
        return fail(SSD_ERR_UNSUPPORTED, "B <= 65535, S <= 1048560 and C < 2^31 required");
    if (dtype != SSD_F32 && dtype != SSD_F16 && dtype != SSD_BF16)
        return fail(SSD_ERR_INVALID_ARG, "unknown dtype code %d", dtype);
    if (!x || !w || !out) return fail(SSD_ERR_INVALID_ARG, "x, w and out are required");
    if (!aligned(x, 16) || !aligned(out, 16)) return fail(SSD_ERR_UNSUPPORTED, "x and out must be 16-byte aligned");
    cudaError_t e = ssd::launch_conv_tokens((int)B, (int)S, (int)C, (int)W, dtype, x, w, bias, silu, out,
                                            static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "causal_conv1d_tokens");
    return ok();
}

ssd_status ssd_causal_conv1d(int64_t B, int64_t D, int64_t S, int64_t W, int32_t dtype, const void *x,
                             const float *w, const float *bias, int32_t silu, void *out, void *stream) {
    if (B <= 0 || D <= 0 || S <= 0 || W <= 0)
        return fail(SSD_ERR_INVALID_ARG, "B, D, S, W must be > 0 (B=%lld D=%lld S=%lld W=%lld)", (long long)B,
                    (long long)D, (long long)S, (long long)W);
    if (W > 8) return fail(SSD_ERR_UNSUPPORTED, "W must be <= 8 (got %lld)", (long long)W);
    if (B > 65535 || D > 65535 || S > 0x7fffffffLL - 1024)
        return fail(SSD_ERR_UNSUPPORTED, "B, D <= 65535 and S < 2^31 required");
    if (dtype != SSD_F32 && dtype != SSD_F16 && dtype != SSD_BF16)
        return fail(SSD_ERR_INVALID_ARG, "unknown dtype code %d", dtype);
    if (!x || !w || !out) return fail(SSD_ERR_INVALID_ARG, "x, w and out are required");
    cudaError_t e = ssd::launch_causal_conv1d((int)B, (int)D, (int)S, (int)W, dtype, x, w, bias, silu, out,
                                              static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "causal_conv1d");
    return ok();
}

ssd_status ssd_gated_rmsnorm(int64_t rows, int64_t D, int64_t groups, float eps, int32_t dtype, const void *x,
                             const void *z, const float *w, void *out, void *stream) {
    if (rows <= 0 || D <= 0 || groups <= 0)
        return fail(SSD_ERR_INVALID_ARG, "rows, D, groups must be > 0");
    if (D % groups != 0)
        return fail(SSD_ERR_INVALID_ARG, "D (%lld) must be a multiple of groups (%lld)", (long long)D,
                    (long long)groups);
    if (!(eps >= 0.f)) return fail(SSD_ERR_INVALID_ARG, "eps must be >= 0");
    if (D > 0x7fffffffLL || rows * groups > 0x7fffffffLL * 8LL)
        return fail(SSD_ERR_UNSUPPORTED, "D < 2^31 and rows * groups < 2^34 required");
    if (dtype != SSD_F32 && dtype != SSD_F16 && dtype != SSD_BF16)
        return fail(SSD_ERR_INVALID_ARG, "unknown dtype code %d", dtype);
    if (!x || !z || !w || !out) return fail(SSD_ERR_INVALID_ARG, "x, z, w and out are required");
    cudaError_t e = ssd::launch_gated_rmsnorm(rows, (int)D, (int)groups, eps, dtype, x, z, w, out,
                                              static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "gated_rmsnorm");
    return ok();
}

ssd_status ssd_decode_step(const ssd_decode_args *a, void *stream) {
    if (!a) return fail(SSD_ERR_INVALID_ARG, "args is NULL");
    if (a->B <= 0 || a->H <= 0 || a->P <= 0 || a->N <= 0 || a->G <= 0)
        return fail(SSD_ERR_INVALID_ARG, "every dim must be > 0 (B=%lld H=%lld P=%lld N=%lld G=%lld)",
                    (long long)a->B, (long long)a->H, (long long)a->P, (long long)a->N, (long long)a->G);
    if (a->H % a->G != 0)
        return fail(SSD_ERR_INVALID_ARG, "H (%lld) must be a multiple of G (%lld)", (long long)a->H,
                    (long long)a->G);
    if (a->N > 128) return fail(SSD_ERR_UNSUPPORTED, "N must be <= 128 (got %lld)", (long long)a->N);
    if (a->B * a->H > 0x7fffffffLL) return fail(SSD_ERR_UNSUPPORTED, "B*H must be < 2^31");
    if (a->x_dtype != SSD_F32 && a->x_dtype != SSD_F16 && a->x_dtype != SSD_BF16)
        return fail(SSD_ERR_INVALID_ARG, "unknown dtype code %d", a->x_dtype);
    if (!(a->dt_min <= a->dt_max) || isnan(a->dt_min) || isnan(a->dt_max))
        return fail(SSD_ERR_INVALID_ARG, "dt_limit must satisfy dt_min <= dt_max");
    if (!a->x || !a->dt || !a->A || !a->Bm || !a->Cm || !a->state || !a->y)
        return fail(SSD_ERR_INVALID_ARG, "x, dt, A, B, C, state and y are required");
    ssd::DecodeParams p;
    p.B = (int)a->B; p.H = (int)a->H; p.P = (int)a->P; p.N = (int)a->N; p.G = (int)a->G;
    p.x = a->x; p.dt = a->dt; p.A = a->A; p.Bm = a->Bm; p.Cm = a->Cm; p.D = a->D; p.z = a->z;
    p.dt_bias = a->dt_bias; p.state = a->state; p.y = a->y;
    p.dt_softplus = a->dt_softplus ? 1 : 0;
    p.has_limit = !(a->dt_min == 0.f && isinf(a->dt_max) && a->dt_max > 0.f);
    p.dt_min = a->dt_min; p.dt_max = a->dt_max;
    cudaError_t e = ssd::launch_decode_step(p, a->x_dtype, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "decode step");
    return ok();
}

ssd_status ssd_segment_log_decay(const ssd_fwd_args *a, float *log_decay, void *stream) {
    ssd_status st = check_shape(a);
    if (st != SSD_OK) return st;
    if (!a->dt || !a->A) return fail(SSD_ERR_INVALID_ARG, "dt and A are required");
    if (!log_decay) return fail(SSD_ERR_INVALID_ARG, "log_decay is required");
    cudaError_t e = ssd::launch_segment_log_decay(make_params(a), log_decay, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "segment_log_decay");
    return ok();
}

ssd_status ssd_state_fold(int64_t nseg, int64_t B, int64_t H, int64_t P, int64_t N, const float *log_decay,
                          const float *states, float *out, void *stream) {
    if (nseg < 0 || B <= 0 || H <= 0 || P <= 0 || N <= 0)
        return fail(SSD_ERR_INVALID_ARG, "nseg >= 0 and B, H, P, N > 0 required");
    if (B * H > 0x7fffffffLL || P * N > 0x7fffffffLL || nseg > 0x7fffffffLL || B * H * P * N > (1LL << 38))
        return fail(SSD_ERR_UNSUPPORTED, "state too large (B*H*P*N <= 2^38)");
    if (!out || (nseg > 0 && (!log_decay || !states)))
        return fail(SSD_ERR_INVALID_ARG, "out (and log_decay, states when nseg > 0) are required");
    cudaError_t e = ssd::launch_state_fold((int)nseg, (long long)(B * H), (int)(P * N), log_decay, states, out,
                                           static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "state_fold");
    return ok();
}

ssd_status ssd_chunk_cumsum(const ssd_fwd_args *a, float *dtp, float *cs, void *stream) {
    ssd_status st = check_shape(a);
    if (st != SSD_OK) return st;
    if (!a->dt || !a->A) return fail(SSD_ERR_INVALID_ARG, "dt and A are required");
    if (!dtp || !cs) return fail(SSD_ERR_INVALID_ARG, "dtp and cs are required");
    cudaError_t e = ssd::launch_chunk_cumsum(make_params(a), dtp, cs, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "chunk_cumsum");
    return ok();
}

ssd_status ssd_chunk_state(const ssd_fwd_args *a, const float *dtp, const float *cs, float *states,
                           void *stream) {
    ssd_status st = check_shape(a);
    if (st != SSD_OK) return st;
    if ((st = check_pointers(a, false)) != SSD_OK) return st;
    if (!dtp || !cs || !states) return fail(SSD_ERR_INVALID_ARG, "dtp, cs and states are required");
    const ssd::Params p = make_params(a);
    cudaError_t e = launch_state_step(a, p, dtp, cs, states, nullptr, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "chunk_state");
    return ok();
}

ssd_status ssd_state_passing(const ssd_fwd_args *a, const float *cs, float *states, void *stream) {
    ssd_status st = check_shape(a);
    if (st != SSD_OK) return st;
    if (a->initial_state && !aligned(a->initial_state, 16))
        return fail(SSD_ERR_INVALID_ARG, "initial_state must be 16-byte aligned");
    if (a->final_state && !aligned(a->final_state, 16))
        return fail(SSD_ERR_INVALID_ARG, "final_state must be 16-byte aligned");
    if (!cs || !states) return fail(SSD_ERR_INVALID_ARG, "cs and states are required");
    if (!aligned(states, 16)) return fail(SSD_ERR_INVALID_ARG, "states must be 16-byte aligned");
    cudaError_t e = ssd::launch_state_passing(make_params(a), cs, states, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "state_passing");
    return ok();
}

ssd_status ssd_chunk_scan(const ssd_fwd_args *a, const float *dtp, const float *cs, const float *states,
                          void *stream) {
    ssd_status st = check_shape(a);
    if (st != SSD_OK) return st;
    if ((st = check_pointers(a, true)) != SSD_OK) return st;
    if (!dtp || !cs || !states) return fail(SSD_ERR_INVALID_ARG, "dtp, cs and states are required");
    const ssd::Params p = make_params(a);
    cudaError_t e = launch_scan_step(a, p, dtp, cs, states, nullptr, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "chunk_scan");
    return ok();
}

// ---- end-to-end entry with host buffers ----------------------------------

namespace {

// How ssd_fwd_host cuts a call into slices.  Along the sequence where the plan
// splits exactly at chunk boundaries (the fused plan at N = 64, whose state is
// fp32 throughout, and the chunked plan): every batch row, `ls` tokens of whole
// chunks per slice (the last may be shorter), the fp32 state handed from slice
// to slice through final_state / initial_state, so the results equal one
// ssd_fwd over the whole call bit for bit and every slice has all of the
// call's work units.  Else (the segmented walks at N = 128 choose their
// segments from L) along the batch.
constexpr int64_t kSeqSlices = 16;
struct HostSlicing {
    bool seq;
    int64_t n;      // slices
    int64_t per_b;  // batch entries per slice (batch slicing)
    int64_t ls;     // tokens per slice (sequence slicing)
};

// Batch entries per slice: up to 8 slices, and one slice when a per-batch
// stride would break the 256-byte alignment of the device copies.
int64_t host_slice_batch(const ssd_fwd_args *a) {
    const size_t io = io_size(a->x_dtype);
    const size_t strides[] = {(size_t)a->L * a->H * a->P * io, (size_t)a->L * a->H * 4,
                              (size_t)a->L * a->G * a->N * io, (size_t)a->H * a->P * a->N * 4};
    for (size_t st : strides)
        if (st % kAlign != 0) return a->B;
    const int64_t nslices = a->B < 8 ? a->B : 8;
    return (a->B + nslices - 1) / nslices;
}

HostSlicing host_slicing(const ssd_fwd_args *a, int32_t plan) {
    const bool exact = (plan == SSD_PLAN_FUSED && a->N == 64) || plan == SSD_PLAN_CHUNKED;
    // (a 2-D copy's pitch is a batch entry of x: kept well inside the copy engines' limit)
    const bool pitch_ok = (size_t)a->L * a->H * a->P * io_size(a->x_dtype) <= ((size_t)1 << 30);
    if (exact && pitch_ok && a->L >= 2 * (int64_t)a->chunk) {
        int64_t ls = (a->L + kSeqSlices - 1) / kSeqSlices;
        ls = (ls + a->chunk - 1) / a->chunk * a->chunk;
        const int64_t n = (a->L + ls - 1) / ls;
        if (n >= 2) return {true, n, a->B, ls};
    }
    const int64_t per = host_slice_batch(a);
    return {false, (a->B + per - 1) / per, per, a->L};
}

// Device copies of the call's tensors in the workspace.  Batch slicing: each
// tensor whole, in its public layout.  Sequence slicing: per slice a block of
// its own compact tensors [B, tokens of the slice, ...] at xs + s * slice_bytes
// (x, dt, B, C, z, y in that order), plus two fp32 states that carry the
// recurrence from slice to slice.
struct HostLayout {
    HostSlicing sl;
    size_t fwd_ws, x, dt, A, Bm, Cm, D, z, dt_bias, h0, y, fin, nw, total;
    size_t slice_bytes, sx, sdt, sb, sc, sz, sy;  // sequence slicing: offsets within a slice block
    size_t st[2];                                 // sequence slicing: the carried states
};

ssd_fwd_args slice_shape(const ssd_fwd_args *a, int64_t L) {
    ssd_fwd_args o = *a;
    o.L = L;
    return o;
}

HostLayout host_layout(const ssd_fwd_args *a, int32_t plan) {
    const size_t io = io_size(a->x_dtype);
    const size_t nst = (size_t)a->B * a->H * a->P * a->N;
    HostLayout l{};
    l.sl = host_slicing(a, plan);
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off += align_up(bytes); return o; };
    if (l.sl.seq) {
        const ssd_fwd_args o = slice_shape(a, l.sl.ls);
        l.fwd_ws = take(workspace_for(&o, plan));
        const size_t tok = (size_t)a->B * l.sl.ls;  // (batch, token) rows of a full slice
        size_t so = 0;
        auto stake = [&](size_t bytes) { size_t r = so; so += align_up(bytes); return r; };
        l.sx = stake(tok * a->H * a->P * io);
        l.sdt = stake(tok * a->H * 4);
        l.sb = stake(tok * a->G * a->N * io);
        l.sc = stake(tok * a->G * a->N * io);
        l.sz = stake(a->z ? tok * a->H * a->P * io : 0);
        l.sy = stake(tok * a->H * a->P * io);
        l.slice_bytes = so;
        l.x = take(so * l.sl.n);
        l.st[0] = take(nst * 4);
        l.st[1] = take(nst * 4);
    } else {
        const size_t nx = (size_t)a->B * a->L * a->H * a->P;
        const size_t nbc = (size_t)a->B * a->L * a->G * a->N;
        l.fwd_ws = take(workspace_for(a, plan));
        l.x = take(nx * io);
        l.dt = take((size_t)a->B * a->L * a->H * 4);
        l.Bm = take(nbc * io);
        l.Cm = take(nbc * io);
        l.z = take(a->z ? nx * io : 0);
        l.y = take(nx * io);
    }
    l.A = take((size_t)a->H * 4);
    l.D = take(a->D ? (size_t)a->H * 4 : 0);
    l.dt_bias = take(a->dt_bias ? (size_t)a->H * 4 : 0);
    l.h0 = take(a->initial_state ? nst * 4 : 0);
    l.fin = take(a->final_state ? nst * 4 : 0);
    l.nw = take(a->norm_weight ? (size_t)a->H * a->P * 4 : 0);
    l.total = off;
    return l;
}

// The host-buffer pipeline: slices copied in on `in`, computed on the
// caller's stream, copied out on `out`, so that the copies in both directions
// and the kernels of different slices overlap.  One set per device, created on
// first use; `mu` serialises the enqueue sequences of concurrent callers (the
// events are re-recorded per slice).
struct HostPipe {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, copied = nullptr, computed = nullptr, done = nullptr;
};
constexpr int kMaxDevices = 64;
std::mutex g_pipe_mu;
HostPipe g_pipes[kMaxDevices];

cudaError_t host_pipe(HostPipe **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    HostPipe &hp = g_pipes[dev];
    if (!hp.ready) {
        if ((e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking)) != cudaSuccess) return e;
        if ((e = cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking)) != cudaSuccess) return e;
        for (cudaEvent_t *ev : {&hp.start, &hp.copied, &hp.computed, &hp.done})
            if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return e;
        hp.ready = true;
    }
    *out = &hp;
    return cudaSuccess;
}

}  // namespace

ssd_status ssd_fwd_host_workspace_size(const ssd_fwd_args *a, size_t *bytes) {
    int32_t plan = 0;
    ssd_status st = reject_conv(a, "ssd_fwd_host");
    if (st != SSD_OK) return st;
    st = ssd_fwd_resolve_plan(a, &plan);
    if (st != SSD_OK) return st;
    if (!bytes) return fail(SSD_ERR_INVALID_ARG, "bytes is NULL");
    *bytes = host_layout(a, plan).total;
    return ok();
}

ssd_status ssd_fwd_host(const ssd_fwd_args *a, void *stream) {
    int32_t plan = 0;
    ssd_status st = reject_conv(a, "ssd_fwd_host");
    if (st != SSD_OK) return st;
    st = ssd_fwd_resolve_plan(a, &plan);
    if (st != SSD_OK) return st;
    if ((st = check_pointers(a, true)) != SSD_OK) return st;
    const HostLayout l = host_layout(a, plan);
    if (!a->workspace || a->workspace_bytes < l.total)
        return fail(SSD_ERR_WORKSPACE, "workspace of %zu bytes required (%zu given)", l.total,
                    a->workspace ? a->workspace_bytes : (size_t)0);
    if (!aligned(a->workspace, kAlign)) return fail(SSD_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(a->workspace);
    const size_t io = io_size(a->x_dtype);
    // per (batch, token) row: bytes of x / y / z, of dt, of B / C; per batch entry: elements of a state
    const size_t rx = (size_t)a->H * a->P * io, rdt = (size_t)a->H * 4, rbc = (size_t)a->G * a->N * io;
    const size_t est = (size_t)a->H * a->P * a->N;
    // what every slice shares: per-head vectors, the fwd workspace, the plan
    ssd_fwd_args d = *a;
    d.A = reinterpret_cast<const float *>(ws + l.A);
    d.D = a->D ? reinterpret_cast<const float *>(ws + l.D) : nullptr;
    d.dt_bias = a->dt_bias ? reinterpret_cast<const float *>(ws + l.dt_bias) : nullptr;
    d.norm_weight = a->norm_weight ? reinterpret_cast<const float *>(ws + l.nw) : nullptr;
    d.workspace = ws + l.fwd_ws;
    d.plan = plan;
    float *h0 = a->initial_state ? reinterpret_cast<float *>(ws + l.h0) : nullptr;
    float *fin = a->final_state ? reinterpret_cast<float *>(ws + l.fin) : nullptr;
    int64_t per = l.sl.per_b;
    if (l.sl.seq) {
        const ssd_fwd_args o = slice_shape(a, l.sl.ls);
        d.workspace_bytes = workspace_for(&o, plan);
    } else {
        d.x = ws + l.x;
        d.dt = reinterpret_cast<const float *>(ws + l.dt);
        d.Bm = ws + l.Bm;
        d.Cm = ws + l.Cm;
        d.z = a->z ? ws + l.z : nullptr;
        d.y = ws + l.y;
        d.initial_state = h0;
        d.final_state = fin;
        d.workspace_bytes = workspace_for(a, plan);
        if (per < a->B) {  // every slice must take the call's plan
            ssd_fwd_args o = d;
            o.B = per;
            int32_t pl = 0;
            if (ssd_fwd_resolve_plan(&o, &pl) != SSD_OK || pl != plan) per = a->B;
        }
    }
    const int64_t nslices = l.sl.seq ? l.sl.n : (a->B + per - 1) / per;
    std::lock_guard<std::mutex> lock(g_pipe_mu);
    HostPipe *hp = nullptr;
    cudaError_t e = host_pipe(&hp);
    if (e != cudaSuccess) return cuda_fail(e, "creating the copy streams");
    // the copy streams start after the caller's earlier work on `stream`
    if ((e = cudaEventRecord(hp->start, s)) != cudaSuccess) return cuda_fail(e, "event record");
    if ((e = cudaStreamWaitEvent(hp->in, hp->start, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(hp->out, hp->start, 0)) != cudaSuccess)
        return cuda_fail(e, "stream wait");
    auto h2d = [&](void *dst, const void *src, size_t bytes) {
        if (e == cudaSuccess && src && bytes) e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, hp->in);
    };
    auto d2h = [&](void *dst, const void *src, size_t bytes) {
        if (e == cudaSuccess && dst && bytes) e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToHost, hp->out);
    };
    // rows [t0, t0 + n) of every batch entry of a [B, L, row bytes] host tensor <-> a compact
    // [B, n, row bytes] device block: one 2-D copy, a batch entry per 2-D row
    auto h2d_rows = [&](void *dst, const void *src, size_t row, int64_t t0, int64_t n) {
        if (e == cudaSuccess && src && row)
            e = cudaMemcpy2DAsync(dst, n * row, static_cast<const char *>(src) + t0 * row, (size_t)a->L * row, n * row,
                                  (size_t)a->B, cudaMemcpyHostToDevice, hp->in);
    };
    auto d2h_rows = [&](void *dst, const void *src, size_t row, int64_t t0, int64_t n) {
        if (e == cudaSuccess && dst && row)
            e = cudaMemcpy2DAsync(static_cast<char *>(dst) + t0 * row, (size_t)a->L * row, src, n * row, n * row,
                                  (size_t)a->B, cudaMemcpyDeviceToHost, hp->out);
    };
    h2d(ws + l.A, a->A, (size_t)a->H * 4);
    h2d(ws + l.D, a->D, (size_t)a->H * 4);
    h2d(ws + l.dt_bias, a->dt_bias, (size_t)a->H * 4);
    h2d(ws + l.nw, a->norm_weight, (size_t)a->H * a->P * 4);
    h2d(h0, a->initial_state, (size_t)a->B * est * 4);
    ssd_status st2 = SSD_OK;
    for (int64_t si = 0; si < nslices && e == cudaSuccess && st2 == SSD_OK; ++si) {
        ssd_fwd_args o = d;
        int64_t b0 = 0, nb = a->B, t0 = 0, nt = a->L;
        if (l.sl.seq) {
            t0 = si * l.sl.ls;
            nt = a->L - t0 < l.sl.ls ? a->L - t0 : l.sl.ls;
            char *blk = ws + l.x + si * l.slice_bytes;
            o.L = nt;
            o.x = blk + l.sx;
            o.dt = reinterpret_cast<const float *>(blk + l.sdt);
            o.Bm = blk + l.sb;
            o.Cm = blk + l.sc;
            o.z = a->z ? blk + l.sz : nullptr;
            o.y = blk + l.sy;
            // the state entering the slice, and the state it leaves for the next one
            o.initial_state = si == 0 ? h0 : reinterpret_cast<const float *>(ws + l.st[(si - 1) & 1]);
            o.final_state = si + 1 == nslices ? fin : reinterpret_cast<float *>(ws + l.st[si & 1]);
            h2d_rows(const_cast<void *>(o.x), a->x, rx, t0, nt);
            h2d_rows(const_cast<float *>(o.dt), a->dt, rdt, t0, nt);
            h2d_rows(const_cast<void *>(o.Bm), a->Bm, rbc, t0, nt);
            h2d_rows(const_cast<void *>(o.Cm), a->Cm, rbc, t0, nt);
            if (a->z) h2d_rows(const_cast<void *>(o.z), a->z, rx, t0, nt);
        } else {
            b0 = si * per;
            nb = a->B - b0 < per ? a->B - b0 : per;
            const size_t ex = (size_t)a->L * rx, edt = (size_t)a->L * rdt, ebc = (size_t)a->L * rbc;
            o.B = nb;
            o.x = static_cast<const char *>(d.x) + b0 * ex;
            o.dt = reinterpret_cast<const float *>(reinterpret_cast<const char *>(d.dt) + b0 * edt);
            o.Bm = static_cast<const char *>(d.Bm) + b0 * ebc;
            o.Cm = static_cast<const char *>(d.Cm) + b0 * ebc;
            if (o.z) o.z = static_cast<const char *>(d.z) + b0 * ex;
            if (o.initial_state) o.initial_state = d.initial_state + b0 * est;
            o.y = static_cast<char *>(d.y) + b0 * ex;
            if (o.final_state) o.final_state = d.final_state + b0 * est;
            h2d(const_cast<void *>(o.x), static_cast<const char *>(a->x) + b0 * ex, nb * ex);
            h2d(const_cast<float *>(o.dt), reinterpret_cast<const char *>(a->dt) + b0 * edt, nb * edt);
            h2d(const_cast<void *>(o.Bm), static_cast<const char *>(a->Bm) + b0 * ebc, nb * ebc);
            h2d(const_cast<void *>(o.Cm), static_cast<const char *>(a->Cm) + b0 * ebc, nb * ebc);
            if (a->z) h2d(const_cast<void *>(o.z), static_cast<const char *>(a->z) + b0 * ex, nb * ex);
        }
        if (e != cudaSuccess) break;
        if ((e = cudaEventRecord(hp->copied, hp->in)) != cudaSuccess) break;
        if ((e = cudaStreamWaitEvent(s, hp->copied, 0)) != cudaSuccess) break;
        if ((st2 = ssd_fwd(&o, stream)) != SSD_OK) break;
        if ((e = cudaEventRecord(hp->computed, s)) != cudaSuccess) break;
        if ((e = cudaStreamWaitEvent(hp->out, hp->computed, 0)) != cudaSuccess) break;
        if (l.sl.seq) {
            d2h_rows(a->y, o.y, rx, t0, nt);
            if (si + 1 == nslices) d2h(a->final_state, fin, (size_t)a->B * est * 4);
        } else {
            d2h(static_cast<char *>(a->y) + b0 * a->L * rx, o.y, nb * a->L * rx);
            if (a->final_state) d2h(a->final_state + b0 * est, o.final_state, nb * est * 4);
        }
    }
    // join: the call is complete on `stream` once both copy streams are
    cudaError_t ej = cudaEventRecord(hp->computed, hp->in);
    if (ej == cudaSuccess) ej = cudaStreamWaitEvent(s, hp->computed, 0);
    if (ej == cudaSuccess) ej = cudaEventRecord(hp->done, hp->out);
    if (ej == cudaSuccess) ej = cudaStreamWaitEvent(s, hp->done, 0);
    if (st2 != SSD_OK) return st2;
    if (e != cudaSuccess) return cuda_fail(e, "host pipeline copy");
    if (ej != cudaSuccess) return cuda_fail(ej, "joining the copy streams");
    return ok();
}

ssd_status ssd_check_device_error(const ssd_fwd_args *a, void *stream) {
    if (!a || !a->workspace) return fail(SSD_ERR_INVALID_ARG, "args with a workspace required");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    uint32_t word = 0;
    e = cudaMemcpy(&word, a->workspace, sizeof(word), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the error word");
    if (word != 0) return fail(SSD_ERR_TIMEOUT, "device error word 0x%08x", word);
    return ok();
}

}  // extern "C"
