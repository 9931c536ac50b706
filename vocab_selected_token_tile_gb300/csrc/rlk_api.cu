// C ABI of librlk_logp.so: contract validation, argument checks, status
// handling.  Every check that can be made on the host is made here, before
// any launch (PR #289 review excerpt of the vocab-parallel entry point:
// _tile_size and _validate_invocation precede any work; "typed contract"
// commit: incompatible requests are rejected with explicit reasons and never
// served by a silent fallback).
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <initializer_list>
#include <mutex>
#include <string>

#include "rlk_internal.h"
#include "rlk_logp.h"

#define RLK_EXPORT extern "C" __attribute__((visibility("default")))

namespace rlk {

namespace {
thread_local std::string g_last_error;
}

rlk_status fail(rlk_status s, const std::string& why) {
    g_last_error = why;
    return s;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

rlk_status check_contract(const rlk_logp_contract* c) {
    if (!c) return fail(RLK_ERR_INVALID_ARG, "contract is NULL");
    if (c->T < 0) return fail(RLK_ERR_INVALID_ARG, "T must be >= 0");
    if (c->T > ((int64_t)1 << 40)) return fail(RLK_ERR_UNSUPPORTED, "T above 2^40 rows");
    if (c->V_real < 1) return fail(RLK_ERR_INVALID_ARG, "V_real must be >= 1");
    if (c->V_padded < c->V_real) return fail(RLK_ERR_INVALID_ARG, "V_padded must be >= V_real");
    if (c->V_padded > ((int64_t)1 << 31)) return fail(RLK_ERR_UNSUPPORTED, "V_padded above 2^31");
    if (c->num_tiles < 1) return fail(RLK_ERR_INVALID_ARG, "num_tiles must be >= 1");
    if (c->V_padded % c->num_tiles != 0)
        return fail(RLK_ERR_NON_TILEABLE, "vocabulary is not tileable: num_tiles must divide V_padded");
    if (c->virtual_tp != 1 && c->virtual_tp != 2 && c->virtual_tp != 4 && c->virtual_tp != 8)
        return fail(RLK_ERR_UNSUPPORTED, "virtual_tp must be 1, 2, 4 or 8");
    if (c->num_tiles % c->virtual_tp != 0)
        return fail(RLK_ERR_NON_TILEABLE, "shard bounds must be tile-aligned: virtual_tp must divide num_tiles");
    if (c->num_tiles > kMaxTiles) return fail(RLK_ERR_UNSUPPORTED, "num_tiles above 1024");
    if (c->V_padded / c->num_tiles > kMaxTileCols)
        return fail(RLK_ERR_UNSUPPORTED, "tile width V_padded/num_tiles above 16384 columns");
    const int64_t stride = c->row_stride ? c->row_stride : c->V_padded;
    if (stride < c->V_padded) return fail(RLK_ERR_INVALID_ARG, "row_stride must be >= V_padded");
    if (stride % 8 != 0) return fail(RLK_ERR_MISALIGNED, "row_stride must be a multiple of 8 elements (16-byte rows)");
    if (c->mask_mode != RLK_MASK_EXPLICIT && c->mask_mode != RLK_MASK_IGNORE_INDEX)
        return fail(RLK_ERR_INVALID_ARG, "mask_mode must be RLK_MASK_EXPLICIT or RLK_MASK_IGNORE_INDEX");
    if (c->validate != 0 && c->validate != 1) return fail(RLK_ERR_INVALID_ARG, "validate must be 0 or 1");
    if (c->wait_timeout_ns < 0) return fail(RLK_ERR_INVALID_ARG, "wait_timeout_ns must be >= 0");
    return check_planner_env();
}

rlk_status check_common(const rlk_logp_contract* c, const void* logits, const int64_t* targets,
                        const uint8_t* mask, const void* workspace) {
    if (!logits) return fail(RLK_ERR_INVALID_ARG, "logits is NULL");
    if (!aligned16(logits)) return fail(RLK_ERR_MISALIGNED, "logits must be 16-byte aligned");
    if (!targets) return fail(RLK_ERR_INVALID_ARG, "targets is NULL");
    if (c->mask_mode == RLK_MASK_EXPLICIT && !mask)
        return fail(RLK_ERR_INVALID_ARG, "explicit mask mode needs active_mask");
    if (c->mask_mode == RLK_MASK_IGNORE_INDEX && mask)
        return fail(RLK_ERR_INVALID_ARG, "ignore_index mode takes no active_mask (pass NULL)");
    if (!workspace) return fail(RLK_ERR_INVALID_ARG, "workspace is NULL");
    if (!aligned16(workspace)) return fail(RLK_ERR_MISALIGNED, "workspace must be 16-byte aligned");
    return RLK_OK;
}

// dlogits may be the logits buffer itself (in place: the kernels read every
// logit before its gradient overwrites it) or a buffer of its own; any other
// overlap would let one row's gradient land on logits not yet read.
rlk_status check_dlogits_overlap(const void* logits, const void* dlogits, int64_t T, int64_t stride) {
    if (logits == dlogits) return RLK_OK;
    const uint64_t a = reinterpret_cast<uintptr_t>(logits), b = reinterpret_cast<uintptr_t>(dlogits);
    const uint64_t rows = (uint64_t)T, st = (uint64_t)stride;
    const uint64_t span = (st != 0 && rows > (UINT64_MAX / 2) / st) ? UINT64_MAX : rows * st * 2u;
    if ((a < b ? b - a : a - b) < span)
        return fail(RLK_ERR_INVALID_ARG, "dlogits overlaps logits without being the same buffer (only an exact "
                                         "in-place call, dlogits == logits, may share memory)");
    return RLK_OK;
}

// Makes the device that owns `ptr` current for this library's runtime.
rlk_status select_device(const void* ptr) {
    cudaPointerAttributes attr{};
    cudaError_t e = cudaPointerGetAttributes(&attr, ptr);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(RLK_ERR_INVALID_ARG, std::string("the first device operand is not a CUDA pointer: ") +
                                             cudaGetErrorString(e));
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
        return fail(RLK_ERR_INVALID_ARG, "device buffers must be device memory");
    e = cudaSetDevice(attr.device);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("cudaSetDevice: ") + cudaGetErrorString(e));
    return RLK_OK;
}

struct DevPtr {
    const void* ptr;
    const char* name;
};

// Every other pointer a call receives must be device memory of the device
// select_device made current (or managed memory, which that device can
// reach).  Host memory -- pinned or not -- and another GPU's memory fail
// closed here, before any launch, instead of reaching a kernel.  NULL
// entries are optional arguments the caller left out.
rlk_status check_device_ptrs(std::initializer_list<DevPtr> ptrs) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    for (const DevPtr& d : ptrs) {
        if (!d.ptr) continue;
        cudaPointerAttributes attr{};
        e = cudaPointerGetAttributes(&attr, d.ptr);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(RLK_ERR_INVALID_ARG, std::string(d.name) + " is not a CUDA pointer");
        }
        if (attr.type == cudaMemoryTypeManaged) continue;
        if (attr.type != cudaMemoryTypeDevice)
            return fail(RLK_ERR_INVALID_ARG, std::string(d.name) + " must be device memory (it is host memory)");
        if (attr.device != dev)
            return fail(RLK_ERR_INVALID_ARG, std::string(d.name) + " lives on device " + std::to_string(attr.device) +
                                                 ", not on device " + std::to_string(dev) +
                                                 " that holds the first operand");
    }
    return RLK_OK;
}

rlk_status decode_status(uint32_t bits) {
    if (bits & kStatusInternal)
        return fail(RLK_ERR_CUDA, "a streaming kernel found a ring slot holding an unexpected row and stopped");
    if (bits & kStatusTimeout) return fail(RLK_ERR_TIMEOUT, "a bounded device-side wait expired");
    if (bits & kStatusTargetRange) return fail(RLK_ERR_TARGET_RANGE, "an active target lies outside [0, V_real)");
    if (bits & kStatusNonFinite)
        return fail(RLK_ERR_NONFINITE_LSE,
                    "non-finite logsumexp on an active row: its real-vocabulary logits must be finite");
    return RLK_OK;
}

rlk_status read_status(const void* workspace, cudaStream_t stream) {
    uint32_t bits = 0;
    cudaError_t e = cudaMemcpyAsync(&bits, workspace, sizeof(bits), cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("reading the status word: ") + cudaGetErrorString(e));
    return decode_status(bits);
}

rlk_status begin(void* workspace, cudaStream_t stream) {
    cudaError_t e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), stream);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("clearing the status word: ") + cudaGetErrorString(e));
    return RLK_OK;
}

}  // namespace
}  // namespace rlk

using namespace rlk;

RLK_EXPORT rlk_status rlk_logp_check_contract(const rlk_logp_contract* contract) {
    return check_contract(contract);
}

RLK_EXPORT size_t rlk_logp_workspace_size(const rlk_logp_contract* contract) {
    return check_contract(contract) == RLK_OK ? kWorkspaceBytes : 0;
}

RLK_EXPORT rlk_status rlk_logp_fwd(const rlk_logp_contract* c, const void* logits_bf16, const int64_t* targets,
                                   const uint8_t* active_mask, float* logp, float* lse, float* partials,
                                   void* workspace, rlk_stream_t stream) {
    rlk_status s = check_contract(c);
    if (s != RLK_OK) return s;
    if (c->T == 0) return RLK_OK;
    if ((s = check_common(c, logits_bf16, targets, active_mask, workspace)) != RLK_OK) return s;
    if (!logp || !lse) return fail(RLK_ERR_INVALID_ARG, "logp and lse outputs are required");
    if ((s = select_device(logits_bf16)) != RLK_OK) return s;
    if ((s = check_device_ptrs({{targets, "targets"}, {active_mask, "active_mask"}, {logp, "logp"}, {lse, "lse"},
                                {partials, "partials"}, {workspace, "workspace"}})) != RLK_OK)
        return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((s = begin(workspace, st)) != RLK_OK) return s;
    StreamArgs a{};
    a.logits = static_cast<const uint16_t*>(logits_bf16);
    a.targets = targets;
    a.mask = active_mask;
    a.logp = logp;
    a.lse = lse;
    a.partials = partials;
    a.status = static_cast<uint32_t*>(workspace);
    if ((s = launch_stream(*c, kModeFwd, a, st)) != RLK_OK) return s;
    return c->validate ? read_status(workspace, st) : RLK_OK;
}

RLK_EXPORT rlk_status rlk_logp_fwd_entropy(const rlk_logp_contract* c, const void* logits_bf16,
                                           const int64_t* targets, const uint8_t* active_mask, float* logp,
                                           float* lse, float* entropy, void* workspace, rlk_stream_t stream) {
    rlk_status s = check_contract(c);
    if (s != RLK_OK) return s;
    if (c->T == 0) return RLK_OK;
    if ((s = check_common(c, logits_bf16, targets, active_mask, workspace)) != RLK_OK) return s;
    if (!logp || !lse || !entropy) return fail(RLK_ERR_INVALID_ARG, "logp, lse and entropy outputs are required");
    if ((s = select_device(logits_bf16)) != RLK_OK) return s;
    if ((s = check_device_ptrs({{targets, "targets"}, {active_mask, "active_mask"}, {logp, "logp"}, {lse, "lse"},
                                {entropy, "entropy"}, {workspace, "workspace"}})) != RLK_OK)
        return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((s = begin(workspace, st)) != RLK_OK) return s;
    StreamArgs a{};
    a.logits = static_cast<const uint16_t*>(logits_bf16);
    a.targets = targets;
    a.mask = active_mask;
    a.logp = logp;
    a.lse = lse;
    a.entropy = entropy;
    a.status = static_cast<uint32_t*>(workspace);
    if ((s = launch_stream(*c, kModeFwd, a, st)) != RLK_OK) return s;
    return c->validate ? read_status(workspace, st) : RLK_OK;
}

RLK_EXPORT rlk_status rlk_logp_fwd_bwd_entropy(const rlk_logp_contract* c, const void* logits_bf16,
                                               const int64_t* targets, const uint8_t* active_mask,
                                               const float* grad_logp, void* dlogits_bf16, float* logp_out,
                                               float* lse_out, float* entropy_out, void* workspace,
                                               rlk_stream_t stream) {
    rlk_status s = check_contract(c);
    if (s != RLK_OK) return s;
    if (c->T == 0) return RLK_OK;
    if ((s = check_common(c, logits_bf16, targets, active_mask, workspace)) != RLK_OK) return s;
    if (!grad_logp) return fail(RLK_ERR_INVALID_ARG, "grad_logp is NULL");
    if (!dlogits_bf16) return fail(RLK_ERR_INVALID_ARG, "dlogits is NULL");
    if (!aligned16(dlogits_bf16)) return fail(RLK_ERR_MISALIGNED, "dlogits must be 16-byte aligned");
    if ((s = check_dlogits_overlap(logits_bf16, dlogits_bf16, c->T, c->row_stride ? c->row_stride : c->V_padded)) !=
        RLK_OK)
        return s;
    if (!logp_out || !lse_out || !entropy_out)
        return fail(RLK_ERR_INVALID_ARG, "logp_out, lse_out and entropy_out are required");
    if ((s = select_device(logits_bf16)) != RLK_OK) return s;
    if ((s = check_device_ptrs({{targets, "targets"}, {active_mask, "active_mask"}, {grad_logp, "grad_logp"},
                                {dlogits_bf16, "dlogits"}, {logp_out, "logp_out"}, {lse_out, "lse_out"},
                                {entropy_out, "entropy_out"}, {workspace, "workspace"}})) != RLK_OK)
        return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((s = begin(workspace, st)) != RLK_OK) return s;
    StreamArgs a{};
    a.logits = static_cast<const uint16_t*>(logits_bf16);
    a.dlogits = static_cast<uint16_t*>(dlogits_bf16);
    a.targets = targets;
    a.mask = active_mask;
    a.grad = grad_logp;
    a.logp = logp_out;
    a.lse = lse_out;
    a.entropy = entropy_out;
    a.status = static_cast<uint32_t*>(workspace);
    if ((s = launch_stream(*c, kModeFused, a, st)) != RLK_OK) return s;
    return c->validate ? read_status(workspace, st) : RLK_OK;
}

RLK_EXPORT rlk_status rlk_grpo_loss(int64_t T, const float* logp, const float* advantage, const uint8_t* active_mask,
                                    const float* ref_logp, float beta, float* loss, float* grad_logp,
                                    float* active_count, rlk_stream_t stream) {
    if (T < 0) return fail(RLK_ERR_INVALID_ARG, "T must be >= 0");
    if (!loss) return fail(RLK_ERR_INVALID_ARG, "loss output is required");
    if (T > 0 && (!logp || !advantage || !active_mask || !grad_logp))
        return fail(RLK_ERR_INVALID_ARG, "logp, advantage, active_mask and grad_logp are required");
    if (!(beta >= 0.f) || !isfinite(beta)) return fail(RLK_ERR_INVALID_ARG, "beta must be finite and >= 0");
    rlk_status s = select_device(loss);
    if (s != RLK_OK) return s;
    if ((s = check_device_ptrs({{logp, "logp"}, {advantage, "advantage"}, {active_mask, "active_mask"},
                                {ref_logp, "ref_logp"}, {grad_logp, "grad_logp"}, {active_count, "active_count"}})) !=
        RLK_OK)
        return s;
    return launch_grpo_loss(T, logp, advantage, active_mask, ref_logp, beta, loss, grad_logp, active_count,
                            reinterpret_cast<cudaStream_t>(stream));
}

namespace rlk {
namespace {
// Workspace of the fused GRPO step: the status word, N (8 bytes in 256), and
// in ignore_index mode each row's activity for the loss (one byte a row).
constexpr size_t kGrpoCountBytes = 256;
size_t grpo_workspace(const rlk_logp_contract& c) {
    return kWorkspaceBytes + kGrpoCountBytes + ((size_t)c.T + 255) / 256 * 256;
}
}  // namespace
}  // namespace rlk

RLK_EXPORT size_t rlk_grpo_fused_workspace_size(const rlk_logp_contract* c) {
    return check_contract(c) == RLK_OK ? grpo_workspace(*c) : 0;
}

RLK_EXPORT rlk_status rlk_grpo_fused_step(const rlk_logp_contract* c, const void* logits_bf16,
                                          const int64_t* targets, const uint8_t* active_mask, const float* advantage,
                                          const float* ref_logp, float beta, void* dlogits_bf16, float* logp_out,
                                          float* lse_out, float* grad_out, float* entropy_out, float* loss,
                                          float* active_count, void* workspace, rlk_stream_t stream) {
    rlk_status s = check_contract(c);
    if (s != RLK_OK) return s;
    if (!loss) return fail(RLK_ERR_INVALID_ARG, "loss output is required");
    if (!(beta >= 0.f) || !isfinite(beta)) return fail(RLK_ERR_INVALID_ARG, "beta must be finite and >= 0");
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (c->T == 0) {  // no rows: loss 0 (and N = 0)
        if ((s = select_device(loss)) != RLK_OK) return s;
        if ((s = check_device_ptrs({{active_count, "active_count"}})) != RLK_OK) return s;
        return launch_grpo_loss(0, nullptr, nullptr, nullptr, nullptr, beta, loss, nullptr, active_count, st);
    }
    if ((s = check_common(c, logits_bf16, targets, active_mask, workspace)) != RLK_OK) return s;
    if (!advantage) return fail(RLK_ERR_INVALID_ARG, "advantage is NULL");
    if (!dlogits_bf16) return fail(RLK_ERR_INVALID_ARG, "dlogits is NULL");
    if (!aligned16(dlogits_bf16)) return fail(RLK_ERR_MISALIGNED, "dlogits must be 16-byte aligned");
    if ((s = check_dlogits_overlap(logits_bf16, dlogits_bf16, c->T, c->row_stride ? c->row_stride : c->V_padded)) !=
        RLK_OK)
        return s;
    if (!logp_out || !lse_out || !grad_out)
        return fail(RLK_ERR_INVALID_ARG, "logp_out, lse_out and grad_out are required");
    if ((s = select_device(logits_bf16)) != RLK_OK) return s;
    if ((s = check_device_ptrs({{targets, "targets"}, {active_mask, "active_mask"}, {advantage, "advantage"},
                                {ref_logp, "ref_logp"}, {dlogits_bf16, "dlogits"}, {logp_out, "logp_out"},
                                {lse_out, "lse_out"}, {grad_out, "grad_out"}, {entropy_out, "entropy_out"},
                                {loss, "loss"}, {active_count, "active_count"}, {workspace, "workspace"}})) != RLK_OK)
        return s;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("querying the device: ") + cudaGetErrorString(e));
    if ((s = begin(workspace, st)) != RLK_OK) return s;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    auto* n_active = reinterpret_cast<unsigned long long*>(ws + kWorkspaceBytes);
    uint8_t* mask_ws = (c->mask_mode == RLK_MASK_IGNORE_INDEX) ? ws + kWorkspaceBytes + kGrpoCountBytes : nullptr;
    if ((s = launch_grpo_count(c->T, targets, active_mask, c->ignore_index, mask_ws, n_active, sms, st)) != RLK_OK)
        return s;
    StreamArgs a{};
    a.logits = static_cast<const uint16_t*>(logits_bf16);
    a.dlogits = static_cast<uint16_t*>(dlogits_bf16);
    a.targets = targets;
    a.mask = active_mask;
    a.logp = logp_out;
    a.lse = lse_out;
    a.entropy = entropy_out;
    a.status = static_cast<uint32_t*>(workspace);
    a.grpo = 1;
    a.adv = advantage;
    a.ref = ref_logp;
    a.beta = beta;
    a.n_active = n_active;
    a.grad_out = grad_out;
    if ((s = launch_stream(*c, kModeFused, a, st)) != RLK_OK) return s;
    // the loss from this step's logp, in the GRPO loss kernel's fixed order (g is already written)
    if ((s = launch_grpo_loss(c->T, logp_out, advantage, active_mask ? active_mask : mask_ws, ref_logp, beta, loss,
                              nullptr, active_count, st)) != RLK_OK)
        return s;
    return c->validate ? read_status(workspace, st) : RLK_OK;
}

RLK_EXPORT rlk_status rlk_logp_bwd(const rlk_logp_contract* c, const void* logits_bf16, const int64_t* targets,
                                   const uint8_t* active_mask, const float* lse_in, const float* grad_logp,
                                   void* dlogits_bf16, float* logp_out, float* lse_out, void* workspace,
                                   rlk_stream_t stream) {
    rlk_status s = check_contract(c);
    if (s != RLK_OK) return s;
    if (c->T == 0) return RLK_OK;
    if ((s = check_common(c, logits_bf16, targets, active_mask, workspace)) != RLK_OK) return s;
    if (!grad_logp) return fail(RLK_ERR_INVALID_ARG, "grad_logp is NULL");
    if (!dlogits_bf16) return fail(RLK_ERR_INVALID_ARG, "dlogits is NULL");
    if (!aligned16(dlogits_bf16)) return fail(RLK_ERR_MISALIGNED, "dlogits must be 16-byte aligned");
    if ((s = check_dlogits_overlap(logits_bf16, dlogits_bf16, c->T, c->row_stride ? c->row_stride : c->V_padded)) !=
        RLK_OK)
        return s;
    if (lse_in && (logp_out || lse_out))
        return fail(RLK_ERR_INVALID_ARG, "with lse_in the forward outputs logp_out/lse_out must be NULL");
    if (!lse_in && (!logp_out || !lse_out))
        return fail(RLK_ERR_INVALID_ARG, "the fused form (lse_in NULL) needs logp_out and lse_out");
    if ((s = select_device(logits_bf16)) != RLK_OK) return s;
    if ((s = check_device_ptrs({{targets, "targets"}, {active_mask, "active_mask"}, {lse_in, "lse_in"},
                                {grad_logp, "grad_logp"}, {dlogits_bf16, "dlogits"}, {logp_out, "logp_out"},
                                {lse_out, "lse_out"}, {workspace, "workspace"}})) != RLK_OK)
        return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((s = begin(workspace, st)) != RLK_OK) return s;
    StreamArgs a{};
    a.logits = static_cast<const uint16_t*>(logits_bf16);
    a.dlogits = static_cast<uint16_t*>(dlogits_bf16);
    a.targets = targets;
    a.mask = active_mask;
    a.grad = grad_logp;
    a.lse_in = lse_in;
    a.logp = logp_out;
    a.lse = lse_out;
    a.status = static_cast<uint32_t*>(workspace);
    if ((s = launch_stream(*c, lse_in ? kModeBwd : kModeFused, a, st)) != RLK_OK) return s;
    return c->validate ? read_status(workspace, st) : RLK_OK;
}

// ---------------------------------------------------------------- fused lm_head

RLK_EXPORT size_t rlk_logp_lmhead_workspace_size(const rlk_logp_contract* c, int64_t H) {
    if (check_contract(c) != RLK_OK || lmhead_check(*c, H) != RLK_OK) return 0;
    return kWorkspaceBytes + lmhead_bwd_workspace(*c);
}

RLK_EXPORT rlk_status rlk_logp_fused_lmhead(const rlk_logp_contract* c, const void* hidden_bf16, int64_t H,
                                            const void* weight_bf16, const int64_t* targets,
                                            const uint8_t* active_mask, const float* grad_logp, float* logp,
                                            float* lse, void* dhidden_bf16, float* dweight_f32, void* dweight_bf16,
                                            void* workspace, rlk_stream_t stream) {
    rlk_status s = check_contract(c);
    if (s != RLK_OK) return s;
    if ((s = lmhead_check(*c, H)) != RLK_OK) return s;
    if (c->T == 0) return RLK_OK;
    if (!hidden_bf16 || !weight_bf16) return fail(RLK_ERR_INVALID_ARG, "hidden and weight are required");
    if (!aligned16(hidden_bf16) || !aligned16(weight_bf16))
        return fail(RLK_ERR_MISALIGNED, "hidden and weight must be 16-byte aligned");
    if (!targets) return fail(RLK_ERR_INVALID_ARG, "targets is NULL");
    if (c->mask_mode == RLK_MASK_EXPLICIT && !active_mask)
        return fail(RLK_ERR_INVALID_ARG, "explicit mask mode needs active_mask");
    if (c->mask_mode == RLK_MASK_IGNORE_INDEX && active_mask)
        return fail(RLK_ERR_INVALID_ARG, "ignore_index mode takes no active_mask (pass NULL)");
    if (!logp || !lse) return fail(RLK_ERR_INVALID_ARG, "logp and lse outputs are required");
    if (!workspace || !aligned16(workspace)) return fail(RLK_ERR_INVALID_ARG, "workspace must be non-NULL and 16-byte aligned");
    const bool bwd = grad_logp != nullptr;
    if (bwd && (!dhidden_bf16 || (!dweight_f32 && !dweight_bf16)))
        return fail(RLK_ERR_INVALID_ARG, "the backward (grad_logp given) needs dhidden and at least one dweight output");
    if (!bwd && (dhidden_bf16 || dweight_f32 || dweight_bf16))
        return fail(RLK_ERR_INVALID_ARG, "dhidden/dweight are written only when grad_logp is given");
    if (bwd && (!aligned16(dhidden_bf16) || !aligned16(dweight_f32) || !aligned16(dweight_bf16)))
        return fail(RLK_ERR_MISALIGNED, "dhidden and dweight must be 16-byte aligned");
    if ((s = select_device(hidden_bf16)) != RLK_OK) return s;
    if ((s = check_device_ptrs({{weight_bf16, "weight"}, {targets, "targets"}, {active_mask, "active_mask"},
                                {grad_logp, "grad_logp"}, {logp, "logp"}, {lse, "lse"}, {dhidden_bf16, "dhidden"},
                                {dweight_f32, "dweight_f32"}, {dweight_bf16, "dweight_bf16"},
                                {workspace, "workspace"}})) != RLK_OK)
        return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((s = begin(workspace, st)) != RLK_OK) return s;
    uint32_t* status = static_cast<uint32_t*>(workspace);
    void* ws = static_cast<unsigned char*>(workspace) + kWorkspaceBytes;
    if (bwd)
        s = launch_lmhead_bwd(*c, hidden_bf16, H, weight_bf16, targets, active_mask, grad_logp, logp, lse,
                              dhidden_bf16, dweight_f32, dweight_bf16, ws, status, st);
    else
        s = launch_lmhead_fwd(*c, hidden_bf16, H, weight_bf16, targets, active_mask, logp, lse, ws, status, st);
    if (s != RLK_OK) return s;
    return c->validate ? read_status(workspace, st) : RLK_OK;
}

RLK_EXPORT rlk_status rlk_logp_fused_lmhead_bwd(const rlk_logp_contract* c, const void* hidden_bf16, int64_t H,
                                                const void* weight_bf16, const int64_t* targets,
                                                const uint8_t* active_mask, const float* lse_in,
                                                const float* grad_logp, void* dhidden_bf16, float* dweight_f32,
                                                void* dweight_bf16, void* workspace, rlk_stream_t stream) {
    rlk_status s = check_contract(c);
    if (s != RLK_OK) return s;
    if ((s = lmhead_check(*c, H)) != RLK_OK) return s;
    if (c->T == 0) return RLK_OK;
    if (!hidden_bf16 || !weight_bf16) return fail(RLK_ERR_INVALID_ARG, "hidden and weight are required");
    if (!aligned16(hidden_bf16) || !aligned16(weight_bf16))
        return fail(RLK_ERR_MISALIGNED, "hidden and weight must be 16-byte aligned");
    if (!targets) return fail(RLK_ERR_INVALID_ARG, "targets is NULL");
    if (c->mask_mode == RLK_MASK_EXPLICIT && !active_mask)
        return fail(RLK_ERR_INVALID_ARG, "explicit mask mode needs active_mask");
    if (c->mask_mode == RLK_MASK_IGNORE_INDEX && active_mask)
        return fail(RLK_ERR_INVALID_ARG, "ignore_index mode takes no active_mask (pass NULL)");
    if (!lse_in || !grad_logp) return fail(RLK_ERR_INVALID_ARG, "lse_in and grad_logp are required");
    if (!dhidden_bf16 || (!dweight_f32 && !dweight_bf16))
        return fail(RLK_ERR_INVALID_ARG, "dhidden and at least one dweight output are required");
    if (!aligned16(dhidden_bf16) || !aligned16(dweight_f32) || !aligned16(dweight_bf16))
        return fail(RLK_ERR_MISALIGNED, "dhidden and dweight must be 16-byte aligned");
    if (!workspace || !aligned16(workspace)) return fail(RLK_ERR_INVALID_ARG, "workspace must be non-NULL and 16-byte aligned");
    if ((s = select_device(hidden_bf16)) != RLK_OK) return s;
    if ((s = check_device_ptrs({{weight_bf16, "weight"}, {targets, "targets"}, {active_mask, "active_mask"},
                                {lse_in, "lse_in"}, {grad_logp, "grad_logp"}, {dhidden_bf16, "dhidden"},
                                {dweight_f32, "dweight_f32"}, {dweight_bf16, "dweight_bf16"},
                                {workspace, "workspace"}})) != RLK_OK)
        return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((s = begin(workspace, st)) != RLK_OK) return s;
    if ((s = launch_lmhead_bwd_given_lse(*c, hidden_bf16, H, weight_bf16, targets, active_mask, grad_logp, lse_in,
                                         dhidden_bf16, dweight_f32, dweight_bf16,
                                         static_cast<unsigned char*>(workspace) + kWorkspaceBytes,
                                         static_cast<uint32_t*>(workspace), st)) != RLK_OK)
        return s;
    return c->validate ? read_status(workspace, st) : RLK_OK;
}

RLK_EXPORT rlk_status rlk_logp_fused_lmhead_keep(const rlk_logp_contract* c, const void* hidden_bf16, int64_t H,
                                                 const void* weight_bf16, const int64_t* targets,
                                                 const uint8_t* active_mask, float* logp, float* lse,
                                                 float* logits_f32, void* workspace, rlk_stream_t stream) {
    rlk_status s = check_contract(c);
    if (s != RLK_OK) return s;
    if ((s = lmhead_check(*c, H)) != RLK_OK) return s;
    if (c->T == 0) return RLK_OK;
    if (!hidden_bf16 || !weight_bf16) return fail(RLK_ERR_INVALID_ARG, "hidden and weight are required");
    if (!aligned16(hidden_bf16) || !aligned16(weight_bf16))
        return fail(RLK_ERR_MISALIGNED, "hidden and weight must be 16-byte aligned");
    if (!targets) return fail(RLK_ERR_INVALID_ARG, "targets is NULL");
    if (c->mask_mode == RLK_MASK_EXPLICIT && !active_mask)
        return fail(RLK_ERR_INVALID_ARG, "explicit mask mode needs active_mask");
    if (c->mask_mode == RLK_MASK_IGNORE_INDEX && active_mask)
        return fail(RLK_ERR_INVALID_ARG, "ignore_index mode takes no active_mask (pass NULL)");
    if (!logp || !lse) return fail(RLK_ERR_INVALID_ARG, "logp and lse outputs are required");
    if (!logits_f32) return fail(RLK_ERR_INVALID_ARG, "logits_f32 is NULL");
    if (!aligned16(logits_f32)) return fail(RLK_ERR_MISALIGNED, "logits_f32 must be 16-byte aligned");
    if (!workspace || !aligned16(workspace)) return fail(RLK_ERR_INVALID_ARG, "workspace must be non-NULL and 16-byte aligned");
    if ((s = select_device(hidden_bf16)) != RLK_OK) return s;
    if ((s = check_device_ptrs({{weight_bf16, "weight"}, {targets, "targets"}, {active_mask, "active_mask"},
                                {logp, "logp"}, {lse, "lse"}, {logits_f32, "logits_f32"},
                                {workspace, "workspace"}})) != RLK_OK)
        return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((s = begin(workspace, st)) != RLK_OK) return s;
    if ((s = launch_lmhead_fwd_keep(*c, hidden_bf16, H, weight_bf16, targets, active_mask, logp, lse, logits_f32,
                                    static_cast<unsigned char*>(workspace) + kWorkspaceBytes,
                                    static_cast<uint32_t*>(workspace), st)) != RLK_OK)
        return s;
    return c->validate ? read_status(workspace, st) : RLK_OK;
}

RLK_EXPORT rlk_status rlk_logp_fused_lmhead_bwd_kept(const rlk_logp_contract* c, const void* hidden_bf16, int64_t H,
                                                     const void* weight_bf16, const int64_t* targets,
                                                     const uint8_t* active_mask, const float* lse_in,
                                                     const float* logits_f32, const float* grad_logp,
                                                     void* dhidden_bf16, float* dweight_f32, void* dweight_bf16,
                                                     void* workspace, rlk_stream_t stream) {
    rlk_status s = check_contract(c);
    if (s != RLK_OK) return s;
    if ((s = lmhead_check(*c, H)) != RLK_OK) return s;
    if (c->T == 0) return RLK_OK;
    if (!hidden_bf16 || !weight_bf16) return fail(RLK_ERR_INVALID_ARG, "hidden and weight are required");
    if (!aligned16(hidden_bf16) || !aligned16(weight_bf16))
        return fail(RLK_ERR_MISALIGNED, "hidden and weight must be 16-byte aligned");
    if (!targets) return fail(RLK_ERR_INVALID_ARG, "targets is NULL");
    if (c->mask_mode == RLK_MASK_EXPLICIT && !active_mask)
        return fail(RLK_ERR_INVALID_ARG, "explicit mask mode needs active_mask");
    if (c->mask_mode == RLK_MASK_IGNORE_INDEX && active_mask)
        return fail(RLK_ERR_INVALID_ARG, "ignore_index mode takes no active_mask (pass NULL)");
    if (!lse_in || !grad_logp) return fail(RLK_ERR_INVALID_ARG, "lse_in and grad_logp are required");
    if (!logits_f32) return fail(RLK_ERR_INVALID_ARG, "logits_f32 is NULL");
    if (!aligned16(logits_f32)) return fail(RLK_ERR_MISALIGNED, "logits_f32 must be 16-byte aligned");
    if (!dhidden_bf16 || (!dweight_f32 && !dweight_bf16))
        return fail(RLK_ERR_INVALID_ARG, "dhidden and at least one dweight output are required");
    if (!aligned16(dhidden_bf16) || !aligned16(dweight_f32) || !aligned16(dweight_bf16))
        return fail(RLK_ERR_MISALIGNED, "dhidden and dweight must be 16-byte aligned");
    if (!workspace || !aligned16(workspace)) return fail(RLK_ERR_INVALID_ARG, "workspace must be non-NULL and 16-byte aligned");
    if ((s = select_device(hidden_bf16)) != RLK_OK) return s;
    if ((s = check_device_ptrs({{weight_bf16, "weight"}, {targets, "targets"}, {active_mask, "active_mask"},
                                {lse_in, "lse_in"}, {logits_f32, "logits_f32"}, {grad_logp, "grad_logp"},
                                {dhidden_bf16, "dhidden"}, {dweight_f32, "dweight_f32"},
                                {dweight_bf16, "dweight_bf16"}, {workspace, "workspace"}})) != RLK_OK)
        return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((s = begin(workspace, st)) != RLK_OK) return s;
    if ((s = launch_lmhead_bwd_kept(*c, hidden_bf16, H, weight_bf16, targets, active_mask, grad_logp, lse_in,
                                    logits_f32, dhidden_bf16, dweight_f32, dweight_bf16,
                                    static_cast<unsigned char*>(workspace) + kWorkspaceBytes,
                                    static_cast<uint32_t*>(workspace), st)) != RLK_OK)
        return s;
    return c->validate ? read_status(workspace, st) : RLK_OK;
}

// ---------------------------------------------------------------- vocabulary-parallel shards

namespace rlk {
namespace {

// A shard call's contract is the whole problem's, with virtual_tp = the
// number of shards and row_stride that of the shard's buffer (0 -> Vs).
rlk_status check_shard(const rlk_logp_contract* c, int32_t shard) {
    if (!c) return fail(RLK_ERR_INVALID_ARG, "contract is NULL");
    rlk_logp_contract whole = *c;
    whole.row_stride = 0;
    rlk_status s = check_contract(&whole);
    if (s != RLK_OK) return s;
    if (shard < 0 || shard >= c->virtual_tp) return fail(RLK_ERR_INVALID_ARG, "shard must lie in [0, virtual_tp)");
    const int64_t Vs = c->V_padded / c->virtual_tp;
    if (Vs % 8 != 0)
        return fail(RLK_ERR_MISALIGNED, "every shard must start on a 16-byte boundary: V_padded/virtual_tp must be a "
                                        "multiple of 8");
    const int64_t stride = c->row_stride ? c->row_stride : Vs;
    if (stride < Vs) return fail(RLK_ERR_INVALID_ARG, "row_stride of a shard must be >= V_padded/virtual_tp");
    if (stride % 8 != 0) return fail(RLK_ERR_MISALIGNED, "row_stride must be a multiple of 8 elements (16-byte rows)");
    return RLK_OK;
}

}  // namespace

rlk_status check_shard_contract(const rlk_logp_contract& c, int32_t shard) { return check_shard(&c, shard); }

}  // namespace rlk

RLK_EXPORT rlk_status rlk_logp_check_shard_contract(const rlk_logp_contract* c, int32_t shard) {
    return check_shard(c, shard);
}

RLK_EXPORT size_t rlk_logp_shard_workspace_size(const rlk_logp_contract* c) {
    return check_shard(c, 0) == RLK_OK ? kWorkspaceBytes + shard_workspace(*c) : 0;
}

RLK_EXPORT rlk_status rlk_logp_shard_fwd(const rlk_logp_contract* c, int32_t shard, const void* logits_shard,
                                         const int64_t* targets, const uint8_t* active_mask, float* partials_shard,
                                         float* target_logit, void* workspace, rlk_stream_t stream) {
    rlk_status s = check_shard(c, shard);
    if (s != RLK_OK) return s;
    if (c->T == 0) return RLK_OK;
    if ((s = check_common(c, logits_shard, targets, active_mask, workspace)) != RLK_OK) return s;
    if (!partials_shard || !target_logit)
        return fail(RLK_ERR_INVALID_ARG, "partials_shard and target_logit outputs are required");
    if ((s = select_device(logits_shard)) != RLK_OK) return s;
    if ((s = check_device_ptrs({{targets, "targets"}, {active_mask, "active_mask"}, {partials_shard, "partials_shard"},
                                {target_logit, "target_logit"}, {workspace, "workspace"}})) != RLK_OK)
        return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((s = begin(workspace, st)) != RLK_OK) return s;
    if ((s = launch_shard_fwd(*c, shard, static_cast<const uint16_t*>(logits_shard), targets, active_mask,
                              partials_shard, target_logit, static_cast<unsigned char*>(workspace) + kWorkspaceBytes,
                              static_cast<uint32_t*>(workspace), st)) != RLK_OK)
        return s;
    return c->validate ? read_status(workspace, st) : RLK_OK;
}

RLK_EXPORT rlk_status rlk_logp_fold(const rlk_logp_contract* c, const float* gathered_partials,
                                    const float* gathered_target_logit, const int64_t* targets,
                                    const uint8_t* active_mask, float* logp, float* lse, void* workspace,
                                    rlk_stream_t stream) {
    rlk_status s = check_shard(c, 0);
    if (s != RLK_OK) return s;
    if (c->T == 0) return RLK_OK;
    if (!gathered_partials || !gathered_target_logit)
        return fail(RLK_ERR_INVALID_ARG, "gathered_partials and gathered_target_logit are required");
    if (!targets) return fail(RLK_ERR_INVALID_ARG, "targets is NULL");
    if (c->mask_mode == RLK_MASK_EXPLICIT && !active_mask)
        return fail(RLK_ERR_INVALID_ARG, "explicit mask mode needs active_mask");
    if (c->mask_mode == RLK_MASK_IGNORE_INDEX && active_mask)
        return fail(RLK_ERR_INVALID_ARG, "ignore_index mode takes no active_mask (pass NULL)");
    if (!logp || !lse) return fail(RLK_ERR_INVALID_ARG, "logp and lse outputs are required");
    if (!workspace || !aligned16(workspace)) return fail(RLK_ERR_INVALID_ARG, "workspace must be non-NULL and 16-byte aligned");
    if ((s = select_device(gathered_partials)) != RLK_OK) return s;
    if ((s = check_device_ptrs({{gathered_target_logit, "gathered_target_logit"}, {targets, "targets"},
                                {active_mask, "active_mask"}, {logp, "logp"}, {lse, "lse"},
                                {workspace, "workspace"}})) != RLK_OK)
        return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((s = begin(workspace, st)) != RLK_OK) return s;
    if ((s = launch_gathered_fold(*c, gathered_partials, gathered_target_logit, targets, active_mask, logp, lse,
                                  static_cast<uint32_t*>(workspace), st)) != RLK_OK)
        return s;
    return c->validate ? read_status(workspace, st) : RLK_OK;
}

RLK_EXPORT rlk_status rlk_logp_shard_bwd(const rlk_logp_contract* c, int32_t shard, const void* logits_shard,
                                         const int64_t* targets, const uint8_t* active_mask, const float* lse_in,
                                         const float* grad_logp, void* dlogits_shard, void* workspace,
                                         rlk_stream_t stream) {
    rlk_status s = check_shard(c, shard);
    if (s != RLK_OK) return s;
    if (c->T == 0) return RLK_OK;
    if ((s = check_common(c, logits_shard, targets, active_mask, workspace)) != RLK_OK) return s;
    if (!lse_in || !grad_logp) return fail(RLK_ERR_INVALID_ARG, "lse_in and grad_logp are required");
    if (!dlogits_shard) return fail(RLK_ERR_INVALID_ARG, "dlogits_shard is NULL");
    if (!aligned16(dlogits_shard)) return fail(RLK_ERR_MISALIGNED, "dlogits_shard must be 16-byte aligned");
    if ((s = check_dlogits_overlap(logits_shard, dlogits_shard, c->T,
                                   c->row_stride ? c->row_stride : c->V_padded / c->virtual_tp)) != RLK_OK)
        return s;
    if ((s = select_device(logits_shard)) != RLK_OK) return s;
    if ((s = check_device_ptrs({{targets, "targets"}, {active_mask, "active_mask"}, {lse_in, "lse_in"},
                                {grad_logp, "grad_logp"}, {dlogits_shard, "dlogits_shard"},
                                {workspace, "workspace"}})) != RLK_OK)
        return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((s = begin(workspace, st)) != RLK_OK) return s;
    if ((s = launch_shard_bwd(*c, shard, static_cast<const uint16_t*>(logits_shard), targets, active_mask, lse_in,
                              grad_logp, static_cast<uint16_t*>(dlogits_shard),
                              static_cast<unsigned char*>(workspace) + kWorkspaceBytes, static_cast<uint32_t*>(workspace),
                              st)) != RLK_OK)
        return s;
    return c->validate ? read_status(workspace, st) : RLK_OK;
}

// ---------------------------------------------------------------- allocation-free forward
//
// rlk_logp_fwd_noalloc serves callers that may not allocate device memory
// while they run -- an engine whose memory is reserved up front, a plugin
// that is handed a stream but no allocator, a step that must not call the
// synchronising cudaMalloc.  The forward's only scratch (the 256-byte status
// word area that rlk_logp_fwd takes as `workspace`) lives in this file-scope
// array instead; every GPU that loads the library holds it until exit.

namespace rlk {
namespace {

constexpr size_t kNoAllocScratchBytes = 256;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Process-unique id of the calling thread's current CUDA context (the
// driver never reuses one), so that an address looked up in a context that
// has since been destroyed -- by cudaDeviceReset, say -- is never used again.
rlk_status current_context_id(unsigned long long* id) {
    static std::mutex mu;
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!get_current || !get_id) {
            void* f1 = nullptr;
            void* f2 = nullptr;
            cudaDriverEntryPointQueryResult q1, q2;
            if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
                q1 != cudaDriverEntryPointSuccess ||
                cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
                q2 != cudaDriverEntryPointSuccess)
                return fail(RLK_ERR_CUDA, "cannot resolve cuCtxGetCurrent / cuCtxGetId");
            get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
            get_id = reinterpret_cast<CtxGetIdFn>(f2);
        }
    }
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, id) != CUDA_SUCCESS)
        return fail(RLK_ERR_CUDA, "no current CUDA context");
    return RLK_OK;
}

// Device address of g_noalloc_scratch, looked up (cudaGetSymbolAddress, with
// the device current) once per device and context; in host code the array's
// name is only a host-side stand-in, never a device address.
rlk_status noalloc_scratch(void** out) {
    static std::mutex mu;
    static void* addr[64] = {};
    static unsigned long long ctx_of[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(RLK_ERR_UNSUPPORTED, "device ordinal above 63");
    unsigned long long ctx = 0;
    rlk_status s = current_context_id(&ctx);
    if (s != RLK_OK) return s;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev] || ctx_of[dev] != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return fail(RLK_ERR_CUDA, std::string("cudaGetSymbolAddress of the static scratch: ") +
                                          cudaGetErrorString(e));
        addr[dev] = p;
        ctx_of[dev] = ctx;
    }
    *out = addr[dev];
    return RLK_OK;
}

}  // namespace
}  // namespace rlk

RLK_EXPORT rlk_status rlk_logp_fwd_noalloc(const rlk_logp_contract* c, const void* logits_bf16,
                                           const int64_t* targets, const uint8_t* active_mask, float* logp,
                                           float* lse, float* partials, rlk_stream_t stream) {
    rlk_status s = check_contract(c);
    if (s != RLK_OK) return s;
    if (c->T == 0) return RLK_OK;
    if (kWorkspaceBytes > kNoAllocScratchBytes)
        return fail(RLK_ERR_UNSUPPORTED, "this contract needs more scratch than the 256-byte static array; "
                                         "use rlk_logp_fwd with a workspace");
    if (!logits_bf16) return fail(RLK_ERR_INVALID_ARG, "logits is NULL");
    if ((s = select_device(logits_bf16)) != RLK_OK) return s;
    void* scratch = nullptr;
    if ((s = noalloc_scratch(&scratch)) != RLK_OK) return s;
    if ((s = check_common(c, logits_bf16, targets, active_mask, scratch)) != RLK_OK) return s;
    if (!logp || !lse) return fail(RLK_ERR_INVALID_ARG, "logp and lse outputs are required");
    if ((s = check_device_ptrs({{targets, "targets"}, {active_mask, "active_mask"}, {logp, "logp"}, {lse, "lse"},
                                {partials, "partials"}})) != RLK_OK)
        return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((s = begin(scratch, st)) != RLK_OK) return s;  // the status word starts at zero on every call
    StreamArgs a{};
    a.logits = static_cast<const uint16_t*>(logits_bf16);
    a.targets = targets;
    a.mask = active_mask;
    a.logp = logp;
    a.lse = lse;
    a.partials = partials;
    a.status = static_cast<uint32_t*>(scratch);
    if ((s = launch_stream(*c, kModeFwd, a, st)) != RLK_OK) return s;
    return c->validate ? read_status(scratch, st) : RLK_OK;
}

RLK_EXPORT rlk_status rlk_logp_workspace_status(const void* workspace, rlk_stream_t stream) {
    if (!workspace) return fail(RLK_ERR_INVALID_ARG, "workspace is NULL");
    rlk_status s = select_device(workspace);
    if (s != RLK_OK) return s;
    return read_status(workspace, reinterpret_cast<cudaStream_t>(stream));
}

RLK_EXPORT rlk_status rlk_selftest_bounded_wait(int64_t timeout_ns, void* workspace, rlk_stream_t stream) {
    if (timeout_ns <= 0 || timeout_ns > 10000000000ll)
        return fail(RLK_ERR_INVALID_ARG, "timeout_ns must be in (0, 10 s]");
    if (!workspace) return fail(RLK_ERR_INVALID_ARG, "workspace is NULL");
    if (!aligned16(workspace)) return fail(RLK_ERR_MISALIGNED, "workspace must be 16-byte aligned");
    rlk_status s = select_device(workspace);
    if (s != RLK_OK) return s;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if ((s = begin(workspace, st)) != RLK_OK) return s;
    if ((s = launch_selftest_wait((uint64_t)timeout_ns, static_cast<uint32_t*>(workspace), st)) != RLK_OK) return s;
    return read_status(workspace, st);
}

RLK_EXPORT const char* rlk_status_string(rlk_status s) {
    switch (s) {
        case RLK_OK: return "RLK_OK";
        case RLK_ERR_INVALID_ARG: return "RLK_ERR_INVALID_ARG";
        case RLK_ERR_UNSUPPORTED: return "RLK_ERR_UNSUPPORTED";
        case RLK_ERR_NON_TILEABLE: return "RLK_ERR_NON_TILEABLE";
        case RLK_ERR_MISALIGNED: return "RLK_ERR_MISALIGNED";
        case RLK_ERR_TARGET_RANGE: return "RLK_ERR_TARGET_RANGE";
        case RLK_ERR_NONFINITE_LSE: return "RLK_ERR_NONFINITE_LSE";
        case RLK_ERR_TIMEOUT: return "RLK_ERR_TIMEOUT";
        case RLK_ERR_CUDA: return "RLK_ERR_CUDA";
    }
    return "RLK_ERR_UNKNOWN";
}

RLK_EXPORT const char* rlk_last_error_message(void) { return g_last_error.c_str(); }
