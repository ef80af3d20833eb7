// Host side of the persistent decode step (kernel in k_decode_step.cuh): the phase table, the
// shared-memory plan, the attention split and the cooperative launch.
#include <algorithm>
#include <cstdlib>
#include <vector>

#include "k_decode_step.cuh"

namespace lcx {
namespace step_detail {
const void *step_kernel_q4(int hd, int g);
const void *step_kernel_q8(int hd, int g);

namespace {

constexpr int kSlotTarget = 36 * 1024;   // stage size the plan aims for (about 32 KB of weights)

// stage plan of one matrix for ring slots of at most `cap` bytes (the largest tps that fits;
// SwiGLU stages keep at least 2 tasks: the gate and up halves of a feature quad)
StagePlan plan_for(const QMat &W, bool swiglu, int cap) {
    StagePlan pl{};
    pl.quad_bytes = (int)W.quad_bytes();
    const int min_tps = swiglu ? 2 : 1;
    auto bytes = [&](int tps) { return (tps * pl.quad_bytes + 127) / 128 * 128; };
    pl.tps = 4;
    while (pl.tps > min_tps && bytes(pl.tps) > cap) pl.tps /= 2;
    pl.stage_bytes = bytes(pl.tps);
    pl.slots = 0;
    pl.x_bytes = 0;
    pl.smem = 0;
    return pl;
}

StepPhase phase_for(const QMat &W, bool swiglu, int n_tasks, GemvIn in, int cap) {
    StepPhase P{};
    P.p.w = W.w;
    P.p.N = W.N;
    P.p.nb = W.nb;
    P.p.K = W.K;
    P.p.n_tasks = n_tasks;
    P.p.T = 1;
    P.p.in = in;
    P.pl = plan_for(W, swiglu, cap);
    P.n_stages = (n_tasks + P.pl.tps - 1) / P.pl.tps;
    return P;
}

double stored_bytes(const QMat &W, int rows, int k_logical) {
    return (double)rows * ((k_logical + 31) / 32) * (W.type == Q4 ? 18.0 : 34.0);
}

}  // namespace
}  // namespace step_detail

cudaError_t decode_step_prepare(DecodeStep &ds, const DevLayer *layers, int n_layer, const QMat &head,
                                const float *output_norm, const FwdArgs &a) {
    using namespace step_detail;
    ds.tried = true;
    ds.ok = false;
    {
        const char *e = getenv("LCX_DECODE_STEP");   // LCX_DECODE_STEP=0: separate launches instead
        if (e && e[0] == '0') return cudaSuccess;
    }
    const int ql = layers[0].qkv.type, G = a.H / a.KV;
    if (head.type != Q8 || a.KV > 48) return cudaSuccess;   // per-head counters: 48 in the sync block
    const void *kern = ql == Q4 ? step_kernel_q4(a.hd, G) : ql == Q8 ? step_kernel_q8(a.hd, G) : nullptr;
    if (!kern) return cudaSuccess;

    // phases and the slot size: every stage must fit one slot
    int cap = kSlotTarget;
    for (int pass = 0; pass < 2; ++pass) {
        int need = 0;
        for (int l = 0; l < n_layer; ++l) {
            const DevLayer &D = layers[l];
            need = std::max(need, plan_for(D.qkv, false, cap).stage_bytes);
            need = std::max(need, plan_for(D.wo, false, cap).stage_bytes);
            need = std::max(need, plan_for(D.gateup, true, cap).stage_bytes);
            need = std::max(need, plan_for(D.down, false, cap).stage_bytes);
        }
        need = std::max(need, plan_for(head, false, cap).stage_bytes);
        if (need <= cap) break;
        cap = need;
    }
    std::vector<StepPhase> ph;
    int max_nb = 0, slot = 0;
    for (int l = 0; l < n_layer; ++l) {
        const DevLayer &D = layers[l];
        ph.push_back(phase_for(D.qkv, false, (D.qkv.N + 3) / 4, GemvIn{a.x, nullptr, D.attn_norm}, cap));
        ph.push_back(phase_for(D.wo, false, (D.wo.N + 3) / 4, GemvIn{a.o32, nullptr, nullptr}, cap));
        ph.push_back(phase_for(D.gateup, true, (a.F + 1) / 2, GemvIn{a.x, nullptr, D.ffn_norm}, cap));
        ph.push_back(phase_for(D.down, false, (D.down.N + 3) / 4, GemvIn{a.h32, nullptr, nullptr}, cap));
        for (const QMat *W : {&D.qkv, &D.wo, &D.gateup, &D.down}) max_nb = std::max(max_nb, W->nb);
    }
    ph.push_back(phase_for(head, false, (head.N + 3) / 4, GemvIn{a.x, nullptr, output_norm}, cap));
    max_nb = std::max(max_nb, head.nb);
    for (const StepPhase &P : ph) {
        slot = std::max(slot, P.pl.stage_bytes);
        if (gemv_map(P.pl.tps, P.p.nb).NBT > 2) return cudaSuccess;   // rows wider than 16384: separate launches
    }

    // shared memory: staged activations (or attention scratch), then the ring and its barriers
    int dev = 0, optin = 0, n_sm = 0, coop = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    if (!coop) return cudaSuccess;
    cudaFuncAttributes fa{};
    cudaError_t e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    const int x_bytes =
        (std::max<int>((int)stage_bytes_per_token(max_nb), attn_scratch_bytes(a.hd, G)) + 127) / 128 * 128;
    // barriers, then the phase table and the attention unit's page ids
    const int bars = kMaxStages * 8 + (int)(ph.size() * sizeof(StepPhase)) + kMaxUnitPages * 4;
    const long room = (long)optin - (long)fa.sharedSizeBytes - x_bytes - bars - 64;
    // 5 slots where they fit: stages are consumed in pairs, so a pair is in flight while one is
    // used; few enough that the CTA's own loads (activations, attention) do not queue behind many
    const int slots = (int)std::min<long>(5, room > 0 ? room / slot : 0);
    if (slots < 3) return cudaSuccess;
    const size_t smem = (size_t)x_bytes + (size_t)slots * slot + bars;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaSuccess;

    e = cudaMalloc(&ds.ph, ph.size() * sizeof(StepPhase));
    if (e == cudaSuccess) e = cudaMemcpy(ds.ph, ph.data(), ph.size() * sizeof(StepPhase), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMalloc(&ds.sync, 256);
    if (e == cudaSuccess) e = cudaMemset(ds.sync, 0, 256);
    if (e != cudaSuccess) {
        decode_step_release(ds);
        return e;
    }
    ds.kern = kern;
    ds.slot_bytes = slot;
    ds.slots = slots;
    ds.x_bytes = x_bytes;
    ds.smem = smem;
    ds.grid = n_sm;   // one CTA per SM: the ring takes most of an SM's shared memory
    ds.n_ph = (int)ph.size();
    ds.weight_bytes = 0;
    const int qw = a.H * a.hd, kvw = a.KV * a.hd;
    for (int l = 0; l < n_layer; ++l) {
        const DevLayer &D = layers[l];
        ds.weight_bytes += stored_bytes(D.qkv, qw + 2 * kvw, a.d) + stored_bytes(D.wo, a.d, qw) +
                           stored_bytes(D.gateup, 2 * a.F, a.d) + stored_bytes(D.down, a.d, a.F);
    }
    ds.head_bytes = stored_bytes(head, a.V, a.d);
    ds.ok = true;
    return cudaSuccess;
}

void decode_step_release(DecodeStep &ds) {
    if (ds.ph) cudaFree(ds.ph);
    if (ds.sync) cudaFree(ds.sync);
    ds.ph = nullptr;
    ds.sync = nullptr;
    ds.ok = false;
}

cudaError_t decode_step_reset(const DecodeStep &ds, const FwdArgs &a, cudaStream_t s) {
    if (!ds.sync) return cudaSuccess;
    cudaError_t e = cudaMemsetAsync(ds.sync, 0, 256, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(a.att_cnt, 0, (size_t)a.KV * sizeof(int32_t), s);
    return e;
}

cudaError_t launch_decode_step(const DecodeStep &ds, const FwdArgs &a, const void *tok_embd, int t_embd,
                               int32_t *amax_dst, int n_att, cudaStream_t s, int64_t &launches) {
    using namespace step_detail;
    if (!ds.ok || a.T != 1 || a.n_out > 1) return cudaErrorInvalidValue;
    StepArgs sa{};
    sa.ph = reinterpret_cast<const StepPhase *>(ds.ph);
    sa.n_ph_all = ds.n_ph;
    sa.slot_bytes = ds.slot_bytes;
    sa.slots = ds.slots;
    sa.x_bytes = ds.x_bytes;
    sa.sync = ds.sync;
    // attention: one (KV head, cell range) unit per CTA at most, ranges of whole 16-cell groups
    int ns = std::max(1, ds.grid / a.KV);
    ns = std::min(ns, (n_att + 15) / 16);
    ns = std::min(ns, std::min(64, a.att_max_split));
    ns = std::max(ns, 1);
    int chunk = (n_att + ns - 1) / ns;
    chunk = (chunk + 15) / 16 * 16;
    ns = (n_att + chunk - 1) / chunk;
    sa.att_ns = ns;
    sa.att_chunk = chunk;
    sa.kvh_quads = (a.H / a.KV + 2) * a.hd / 4;
    sa.tok_embd = reinterpret_cast<const uint8_t *>(tok_embd);
    sa.t_embd = t_embd;   // the ABI type codes equal QType
    sa.amax_dst = amax_dst;
    FwdArgs aa = a;
    void *args[] = {(void *)&sa, (void *)&aa};
    ++launches;
    return cudaLaunchCooperativeKernel(ds.kern, dim3(ds.grid), dim3(256), args, ds.smem, s);
}

}  // namespace lcx
