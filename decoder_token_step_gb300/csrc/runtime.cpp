// runtime.cpp -- the host side of libsyn: model state, weight store, KV cache, frame allocator,
// RoPE cache, the .archdef sequencer with its load-time fusion pass, CUDA-graph replay of decode
// steps, and the C ABI of include/syn.h.
//
// Lifecycle ("Execution contract", cyber.page): load (create, load weights by GGUF name,
// finalize: completeness check, KV cache sized to the maximum context, RoPE cos/sin cache, fusion
// pass), forward (one step or bulk prefill, appending to the KV cache), reset_kv, drop. Errors are
// structured status codes with a message that names the tensor, op, file line or byte count.
#include <algorithm>
#include <array>
#include <cerrno>
#include <climits>
#include <cstdint>
#include <chrono>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <functional>
#include <map>
#include <memory>
#include <new>
#include <set>
#include <sstream>
#include <string>
#include <vector>

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/syn.h"
#include "syn_internal.h"

using namespace syn;

namespace {

struct Error {
    syn_status code;
    std::string msg;
};

#define CUDA_TRY(call)                                                                                   \
    do {                                                                                                 \
        cudaError_t e_ = (call);                                                                         \
        if (e_ != cudaSuccess) throw Error{SYN_E_CUDA, std::string(#call) + ": " + cudaGetErrorString(e_)}; \
    } while (0)

// ---------------------------------------------------------------------------------------------
// Frame allocator ("Execution contract", section "Memory lifecycle / Activations"): a pool of
// device buffers bucketed by exact byte size. Each forward first calls reset(), after which every
// buffer of the previous forward is free again; alloc() hands out the bucket's buffers in order
// and grows the bucket when it runs out. The pool only grows, to the steady-state size. Because a
// forward asks for the same sizes in the same order, it gets the same addresses every time, which
// is what lets a captured decode graph be replayed.
// ---------------------------------------------------------------------------------------------
class FrameAllocator {
  public:
    void *alloc(size_t bytes) {
        auto &bucket = pool_[bytes];
        size_t &cur = cursor_[bytes];
        if (cur == bucket.size()) {
            void *p = nullptr;
            cudaError_t e = cudaMalloc(&p, std::max<size_t>(bytes, 256));
            if (e != cudaSuccess)
                throw Error{SYN_E_OOM, "frame allocator: cudaMalloc of " + std::to_string(bytes) + " bytes failed: " +
                                           cudaGetErrorString(e)};
            bucket.push_back(p);
            held_ += bytes;
        }
        return bucket[cur++];
    }
    void reset() {
        for (auto &c : cursor_) c.second = 0;
    }
    size_t held() const { return held_; }
    ~FrameAllocator() {
        for (auto &b : pool_)
            for (void *p : b.second) cudaFree(p);
    }

  private:
    std::map<size_t, std::vector<void *>> pool_;
    std::map<size_t, size_t> cursor_;
    size_t held_ = 0;
};

struct DevTensor {
    std::string name;
    int dtype = 0;
    int64_t ne[2] = {1, 1};
    int n_dims = 1;
    void *mem = nullptr;  // single allocation: codes, then scales
    size_t bytes = 0;
    DevMatrix mat;
    const void *tc_planes = nullptr;   // resident tensor-core operand planes (option tc_planes)
    const float *vec() const { return reinterpret_cast<const float *>(mat.codes); }
};

struct Node {
    std::string what;
    int launches = 1;
    std::function<void(cudaStream_t)> run;
    std::string kind = "other";               // profile category
    std::function<double(int)> bytes;         // algorithmic bytes at a given position (optional)
    double flops = 0;                         // arithmetic of a bulk matmul (profile only)
    std::function<double(int)> flops_at;      // arithmetic at a given position (optional, profile only)
};

Node make_node(std::string what, int launches, std::function<void(cudaStream_t)> run) {
    Node n;
    n.what = std::move(what);
    n.launches = launches;
    n.run = std::move(run);
    return n;
}

struct ProfEntry {
    int64_t launches = 0;
    double ms = 0.0;
    double bytes = 0.0;
    double flops = 0.0;
};

struct Plan {
    int n = 0;
    bool fused = false;
    std::vector<Node> nodes;
    std::map<std::string, float *> regs;
    std::set<std::string> folded;  // registers that the fusion pass never materialises
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    bool capture_failed = false;
    int launches() const {
        int s = 0;
        for (auto &nd : nodes) s += nd.launches;
        return s;
    }
    void drop_graph() {
        if (exec) cudaGraphExecDestroy(exec);
        if (graph) cudaGraphDestroy(graph);
        exec = nullptr;
        graph = nullptr;
    }
};

bool is_act(const std::string &op) { return op == "silu" || op == "gelu" || op == "gelu_tanh" || op == "relu"; }
int act_code(const std::string &op) {
    return op == "silu" ? ACT_SILU : op == "gelu" ? ACT_GELU : op == "gelu_tanh" ? ACT_GELU_TANH : ACT_RELU;
}

// registers an op reads (argument kinds from the op signatures; tensors and counts excluded)
std::vector<std::string> reads_of(const Step &s) {
    static const std::map<std::string, std::string> kinds = {
        {"embed", "T"}, {"rms_norm", "RT"}, {"matmul", "RT"}, {"add_bias", "RT"}, {"norm_heads", "RTC"},
        {"rope", "RC"}, {"attention", "RRR"}, {"silu", "R"}, {"gelu", "R"}, {"gelu_tanh", "R"}, {"relu", "R"},
        {"mul", "RR"}, {"add", "RR"}, {"scale", "RS"}, {"copy", "R"}, {"last", "R"}};
    std::vector<std::string> r;
    const std::string &k = kinds.at(s.op);
    for (size_t i = 0; i < k.size() && i < s.args.size(); ++i)
        if (k[i] == 'R') r.push_back(s.args[i]);
    return r;
}

bool reads(const Step &s, const std::string &reg) {
    for (auto &r : reads_of(s))
        if (r == reg) return true;
    return false;
}

}  // namespace

// =============================================================================================
// A conversation's own KV cache on a shared model: its cache buffers, its device position record,
// the host's view of both, and its captured decode plan (the plan's kernels point at the cache).
struct syn_kv {
    syn_model *m = nullptr;
    void *kcache = nullptr, *vcache = nullptr;
    DevState *d_state = nullptr;
    int kv_len = 0, dev_pos = -1, dev_n = -1;
    Plan decode;
    bool decode_ready = false;
    int decode_runs = 0;
    void release() {
        decode.drop_graph();
        cudaFree(kcache);
        cudaFree(vcache);
        cudaFree(d_state);
        kcache = vcache = nullptr;
        d_state = nullptr;
    }
};

struct syn_model {
    std::string err;
    std::string file_arch;
    std::string archdef_sha;   // sha256 of the definition text in effect
    Archdef ad;
    std::map<std::string, std::string> meta;
    int n_layer = 0, n_embd = 0, n_head = 0, n_head_kv = 0, head_dim = 0, window = 0, max_ctx = 0;
    float eps = 1e-6f;
    double rope_base = 10000.0;
    int device = 0, sm_count = 148;
    cudaStream_t stream = nullptr;
    bool own_stream = false;
    bool finalized = false;

    std::map<std::string, DevTensor> tensors;
    std::map<std::string, int> reg_width;
    std::map<std::string, bool> reg_multi;  // holds one row per token (false: one row after `last`)
    int n_vocab = 0;

    void *kcache = nullptr, *vcache = nullptr;   // f32, or f16 with option kv_f16
    size_t kv_es = 4;                            // bytes per cache element
    float2 *rope_cs = nullptr;
    DevState *d_state = nullptr;
    int *d_tokens = nullptr;
    float *arg_v = nullptr;
    int *arg_i = nullptr;
    unsigned *arg_counter = nullptr;
    int arg_blocks = 0;
    unsigned *attn_counters = nullptr;  // [max_ctx][n_head_kv], zero between launches
    FrameAllocator pool;

    int kv_len = 0;
    int dev_pos = -1, dev_n = -1;  // what the host believes DevState holds

    int opt_fusion = 1, opt_graph = 1, opt_timing = 0, opt_splits = 0, opt_profile = 0, opt_tc = 1, opt_attn_tc = 1, opt_kv_f16 = 0, opt_tc_planes = -1;
    std::vector<void *> plane_mem;   // resident tensor-core operand planes (option tc_planes)
    std::map<const void *, const void *> plane_of;   // weight codes -> its planes
    size_t plane_bytes = 0;
    bool planes_decided = false;     // built (or declined) at the first bulk forward
    std::map<std::string, ProfEntry> prof;
    std::vector<cudaEvent_t> prof_ev;
    bool any_fused = false;
    Plan decode;              // cached plan (n == 1)
    bool decode_ready = false;
    int decode_runs = 0;
    const Plan *last_plan = nullptr;  // registers of the last forward (for debug reads)
    Plan bulk;

    cudaEvent_t ev0 = nullptr, ev1 = nullptr;
    // pinned staging ring for the per-step host->device copies (token ids and position), so that
    // a host-driven decode loop never blocks on the GPU; slot reuse waits on the slot's event
    static constexpr int kStageSlots = 16, kStageInts = 32;
    int *h_stage = nullptr;
    int *h_out = nullptr;            // pinned: [0] device error bits, [1] argmax of the last forward
    cudaEvent_t stage_ev[kStageSlots] = {};
    int stage_i = 0;
    syn_timings tm{};
    std::chrono::steady_clock::time_point t_create;

    syn_kv *active = nullptr;          // the selected conversation's state lives in this model
    std::set<syn_kv *> handles;        // every live handle (holding its own state, or the model's own
                                       // while it is the selected one)

    // exchange the per-conversation state of the model with a handle's
    void swap_kv(syn_kv *h) {
        std::swap(kcache, h->kcache);
        std::swap(vcache, h->vcache);
        std::swap(d_state, h->d_state);
        std::swap(kv_len, h->kv_len);
        std::swap(dev_pos, h->dev_pos);
        std::swap(dev_n, h->dev_n);
        std::swap(decode, h->decode);
        std::swap(decode_ready, h->decode_ready);
        std::swap(decode_runs, h->decode_runs);
    }
    // an option changed the decode plan: every conversation rebuilds its plan at its next step
    void invalidate_handle_plans() {
        for (syn_kv *h : handles) {
            h->decode.drop_graph();
            h->decode_ready = false;
        }
    }

    ~syn_model() {
        for (syn_kv *h : handles) {
            h->release();
            h->m = nullptr;   // a later syn_kv_destroy only frees the handle itself
        }
        decode.drop_graph();
        for (auto &t : tensors) cudaFree(t.second.mem);
        drop_planes();
        cudaFree(kcache);
        cudaFree(vcache);
        cudaFree(rope_cs);
        cudaFree(d_state);
        cudaFree(d_tokens);
        cudaFree(arg_v);
        cudaFree(arg_i);
        cudaFree(arg_counter);
        cudaFree(attn_counters);
        if (ev0) cudaEventDestroy(ev0);
        if (ev1) cudaEventDestroy(ev1);
        for (auto &e : stage_ev)
            if (e) cudaEventDestroy(e);
        for (auto &e : prof_ev) cudaEventDestroy(e);
        if (h_stage) cudaFreeHost(h_stage);
        if (h_out) cudaFreeHost(h_out);
        if (own_stream && stream) cudaStreamDestroy(stream);
    }

    // ---------------------------------------------------------------- metadata
    const std::string *meta_arch(const std::string &name) const {
        for (const char *pre : {"", "attention.", "rope."}) {
            auto it = meta.find(ad.arch + "." + pre + name);
            if (it != meta.end()) return &it->second;
        }
        return nullptr;
    }
    int meta_int(const std::string &name, bool required, int dflt = 0) const {
        const std::string *v = meta_arch(name);
        if (!v) {
            if (required) throw Error{SYN_E_INVALID_CONFIG, "missing GGUF metadata key " + ad.arch + "." + name};
            return dflt;
        }
        char *end = nullptr;
        errno = 0;
        const long long x = std::strtoll(v->c_str(), &end, 10);
        if (end == v->c_str() || *end || errno == ERANGE || x < INT32_MIN || x > INT32_MAX)
            throw Error{SYN_E_INVALID_CONFIG, "metadata " + name + " is not a 32-bit integer: '" + *v + "'"};
        return (int)x;
    }
    double meta_double(const std::string &name) const {
        const std::string *v = meta_arch(name);
        if (!v) throw Error{SYN_E_INVALID_CONFIG, "missing GGUF metadata key " + ad.arch + "." + name};
        char *end = nullptr;
        const double x = std::strtod(v->c_str(), &end);
        if (end == v->c_str() || *end || !std::isfinite(x))
            throw Error{SYN_E_INVALID_CONFIG, "metadata " + name + " is not a finite number: '" + *v + "'"};
        return x;
    }

    // ---------------------------------------------------------------- tensors
    std::string expand(const std::string &name, int layer) const {
        std::string r;
        for (size_t i = 0; i < name.size(); ++i) {
            if (name.compare(i, 3, "{i}") == 0) {
                r += std::to_string(layer);
                i += 2;
            } else {
                r += name[i];
            }
        }
        return r;
    }
    // resolve "a | b" (first loaded alternative; "Local inference and architectures", "Rules")
    const DevTensor *find_tensor(const std::string &arg, int layer, std::string *tried = nullptr) const {
        std::stringstream ss(arg);
        std::string part;
        std::string names;
        while (std::getline(ss, part, '|')) {
            size_t a = part.find_first_not_of(" \t"), b = part.find_last_not_of(" \t");
            std::string nm = expand(part.substr(a, b - a + 1), layer);
            auto it = tensors.find(nm);
            if (it != tensors.end()) return &it->second;
            names += (names.empty() ? "" : " | ") + nm;
        }
        if (tried) *tried = names;
        return nullptr;
    }
    const DevTensor &tensor(const Step &st, int argi, int layer) const {
        std::string tried;
        const DevTensor *t = find_tensor(st.args[argi], layer, &tried);
        if (!t)
            throw Error{SYN_E_MISSING_TENSOR, "tensor " + tried + " required by `" + st.op + "` (" + file_arch +
                                                  ".archdef line " + std::to_string(st.line) + ") is not loaded"};
        return *t;
    }
    // The weights of the block's matmuls, which bulk prefill multiplies on the tensor cores.
    std::vector<DevTensor *> bulk_matmul_weights() {
        std::vector<DevTensor *> out;
        for (int l = 0; l < n_layer; ++l)
            for (auto &st : ad.sec[1]) {
                if (st.op != "matmul") continue;
                DevTensor *t = const_cast<DevTensor *>(find_tensor(st.args[1], l));
                if (t && t->mat.K % 8 == 0 && std::find(out.begin(), out.end(), t) == out.end()) out.push_back(t);
            }
        return out;
    }
    void drop_planes() {
        for (auto &kv : tensors) kv.second.tc_planes = nullptr;
        plane_of.clear();
        for (void *p : plane_mem) cudaFree(p);
        plane_mem.clear();
        plane_bytes = 0;
    }
    // Option tc_planes: 1 builds the f16 hi/lo operand planes of every bulk-matmul weight once
    // (4 bytes per weight) so that bulk forwards skip the conversion; -1 does so when they take at
    // most half of the free device memory; 0 converts per bulk forward.
    void build_planes() {
        drop_planes();
        planes_decided = true;
        if (opt_tc_planes == 0 || !opt_tc) return;
        auto ws = bulk_matmul_weights();
        size_t need = 0;
        for (DevTensor *t : ws) need += gemm_tc_planes_bytes(t->mat) + 256;
        if (opt_tc_planes < 0) {
            size_t free_b = 0, total_b = 0;
            if (cudaMemGetInfo(&free_b, &total_b) != cudaSuccess || need > free_b / 2) return;
        }
        for (DevTensor *t : ws) {
            void *p = nullptr;
            const size_t b = gemm_tc_planes_bytes(t->mat);
            if (cudaMalloc(&p, b) != cudaSuccess) {
                drop_planes();
                if (opt_tc_planes < 0) return;
                throw Error{SYN_E_OOM, "tc_planes: cudaMalloc of " + std::to_string(b) + " bytes failed"};
            }
            plane_mem.push_back(p);
            plane_bytes += b;
            CUDA_TRY(launch_dequant_split(t->mat, p, stream));
            t->tc_planes = p;
            plane_of[t->mat.codes] = p;
        }
        CUDA_TRY(cudaStreamSynchronize(stream));
    }
    int head_count(const std::string &name) const {
        int c = meta_int(name, true);
        if (c <= 0) throw Error{SYN_E_INVALID_CONFIG, "metadata " + name + " must be positive"};
        return c;
    }
    bool layer_windowed(int layer) const {
        if (window <= 0) return false;
        if (ad.window_pattern > 0 && layer % ad.window_pattern == ad.window_pattern - 1) return false;
        return true;
    }
    float scale_value(const std::string &a) const {
        const std::string *mv = meta_arch(a);
        return (float)std::strtod(mv ? mv->c_str() : a.c_str(), nullptr);
    }

    // ---------------------------------------------------------------- shape inference
    void infer_shapes() {
        std::map<std::string, int> w;
        std::map<std::string, bool> multi_now;
        auto need_reg = [&](const Step &st, const std::string &r) {
            if (!w.count(r))
                throw Error{SYN_E_SHAPE_MISMATCH, "register " + r + " read before assignment (line " + std::to_string(st.line) + ")"};
            return w[r];
        };
        auto visit = [&](const Step &st, int layer) {
            const std::string &op = st.op;
            int width = 0;
            if (op == "embed") {
                const DevTensor &t = tensor(st, 0, layer);
                if (t.n_dims != 2) throw Error{SYN_E_SHAPE_MISMATCH, "embed: " + t.name + " is not a matrix"};
                width = (int)t.ne[0];
            } else if (op == "matmul") {
                int in = need_reg(st, st.args[0]);
                const DevTensor &t = tensor(st, 1, layer);
                if (t.n_dims != 2 || t.ne[0] != in)
                    throw Error{SYN_E_SHAPE_MISMATCH, "matmul line " + std::to_string(st.line) + ": " + t.name + " has " +
                                                          std::to_string(t.ne[0]) + " in-features, register " + st.args[0] +
                                                          " has width " + std::to_string(in)};
                width = (int)t.ne[1];
            } else if (op == "attention") {
                int wq = need_reg(st, st.args[0]), wk = need_reg(st, st.args[1]), wv = need_reg(st, st.args[2]);
                if (wq != n_head * head_dim || wk != n_head_kv * head_dim || wv != n_head_kv * head_dim)
                    throw Error{SYN_E_SHAPE_MISMATCH, "attention line " + std::to_string(st.line) + ": q/k/v widths " +
                                                          std::to_string(wq) + "/" + std::to_string(wk) + "/" + std::to_string(wv) +
                                                          " do not match heads x head_dim"};
                width = wq;
            } else {
                width = need_reg(st, st.args[0]);
                if (op == "rms_norm" || op == "add_bias") {
                    const DevTensor &t = tensor(st, 1, layer);
                    if (t.ne[0] != width || t.n_dims != 1)
                        throw Error{SYN_E_SHAPE_MISMATCH, op + " line " + std::to_string(st.line) + ": " + t.name + " has " +
                                                              std::to_string(t.ne[0]) + " elements, register has " + std::to_string(width)};
                } else if (op == "norm_heads" || op == "rope") {
                    int nh = head_count(st.args[op == "rope" ? 1 : 2]);
                    if (width % nh || width / nh != head_dim)
                        throw Error{SYN_E_SHAPE_MISMATCH, op + " line " + std::to_string(st.line) + ": width " + std::to_string(width) +
                                                              " is not " + std::to_string(nh) + " heads of " + std::to_string(head_dim)};
                    if (op == "norm_heads") {
                        const DevTensor &t = tensor(st, 1, layer);
                        if (t.ne[0] != head_dim)
                            throw Error{SYN_E_SHAPE_MISMATCH, "norm_heads weight " + t.name + " must have head_dim elements"};
                    }
                } else if (op == "mul" || op == "add") {
                    int w2 = need_reg(st, st.args[1]);
                    if (w2 != width) throw Error{SYN_E_SHAPE_MISMATCH, op + " line " + std::to_string(st.line) + ": widths differ"};
                }
            }
            w[st.dst] = width;
            reg_width[st.dst] = std::max(reg_width[st.dst], width);
            bool multi = op == "embed";
            if (op != "embed" && op != "last")
                for (auto &r : reads_of(st)) multi = multi || multi_now[r];
            multi_now[st.dst] = multi;
            reg_multi[st.dst] = reg_multi[st.dst] || multi;
        };
        for (auto &st : ad.sec[0]) visit(st, -1);
        for (int l = 0; l < n_layer; ++l)
            for (auto &st : ad.sec[1]) visit(st, l);
        for (auto &st : ad.sec[2]) visit(st, -1);
        if (!reg_width.count("logits")) throw Error{SYN_E_SHAPE_MISMATCH, "no logits register"};
        n_vocab = reg_width["logits"];
    }

    // ---------------------------------------------------------------- liveness
    // Is `reg` overwritten before it is read again, looking forward from step idx of section sec
    // (a block wraps around to the next layer, then the epilogue follows)?
    bool dead_after(const std::string &reg, int sec, size_t idx) const {
        std::vector<const Step *> seq;
        const auto &S = ad.sec[sec];
        for (size_t i = idx + 1; i < S.size(); ++i) seq.push_back(&S[i]);
        if (sec == 1) {
            for (size_t i = 0; i <= idx; ++i) seq.push_back(&S[i]);
            for (auto &st : ad.sec[2]) seq.push_back(&st);
        } else if (sec == 0) {
            for (auto &st : ad.sec[1]) seq.push_back(&st);
            for (auto &st : ad.sec[2]) seq.push_back(&st);
        }
        for (const Step *s : seq) {
            if (reads(*s, reg)) return false;
            if (s->assign && s->dst == reg) return true;
        }
        return true;  // never read again
    }

    // ---------------------------------------------------------------- plan building
    struct Ctx {
        int n = 1;
        bool fused = false;
        std::map<std::string, float *> buf;
        std::map<std::string, int> rows;
        std::map<std::string, std::pair<std::string, const float *>> fold_rms;  // h -> (x, w)
        // decode: a post-branch update `x += rms_norm(t, w)` waiting for the next matmul that reads
        // x to take it into its prologue (GemvPre); `at` is where its own node goes
        // if something else reads x first
        struct PendingPre {
            const float *t = nullptr;
            const float *w = nullptr;
            size_t at = 0;
            Node node;
        };
        std::map<std::string, PendingPre> pre;
        std::map<std::string, float *> alt;   // a register's second buffer (x_new is written there)
        float *part = nullptr;
        int splits = 1;
        float *tmp = nullptr;
        // scratch of the tensor-core bulk matmuls (f16 hi/lo planes), shared by every such node of
        // the plan and allocated once the largest need is known
        struct TcScratch {
            size_t x_bytes = 0, w_bytes = 0;
            void *x = nullptr, *w = nullptr;
        };
        std::shared_ptr<TcScratch> tc = std::make_shared<TcScratch>();
        // scratch of the tensor-core prefill attention (f16 hi/lo planes of q and of the cache)
        struct AttnTcScratch {
            size_t q_bytes = 0, kv_bytes = 0;
            void *q = nullptr, *kv = nullptr;
        };
        std::shared_ptr<AttnTcScratch> atc = std::make_shared<AttnTcScratch>();
    };

    int64_t ld(const std::string &r) const { return reg_width.at(r); }

    GemvSeg seg_for(const DevTensor &t, float *out, const std::string &dst) const {
        GemvSeg s;
        s.W = t.mat;
        s.out = out;
        s.ldo = ld(dst);
        return s;
    }

    void emit_matmul(Plan &P, Ctx &c, std::vector<GemvSeg> segs, const std::string &src, int act_gate_up,
                     const std::string &what) {
        GemvParams g;
        for (size_t i = 0; i < segs.size(); ++i) g.seg[i] = segs[i];
        g.nseg = (int)segs.size();
        std::string x = src;
        auto fr = c.fold_rms.find(src);
        if (fr != c.fold_rms.end()) {
            x = fr->second.first;
            g.norm_w = fr->second.second;
            g.eps = eps;
        }
        g.x = c.buf.at(x);
        g.ldx = ld(x);
        g.rows = c.rows.at(x);
        if (act_gate_up) {
            g.gate_up = 1;
            g.act = act_gate_up;
        }
        GemvPre pre;
        auto pp = c.pre.find(x);
        if (pp != c.pre.end() && g.rows == 1 && ld(x) == g.seg[0].W.K) {
            // the pending post-branch update runs in this matmul's prologue; x_new goes to the
            // register's other buffer, which holds x from here on
            float *&other = c.alt[x];
            if (!other) other = static_cast<float *>(pool.alloc((size_t)ld(x) * sizeof(float)));
            pre.t = pp->second.t;
            pre.w = pp->second.w;
            pre.out = other;
            std::swap(c.buf[x], other);
            P.regs[x] = c.buf[x];
            c.pre.erase(pp);
        }
        const int sms = sm_count;
        // algorithmic bytes: every weight byte once (codes + block scales), the input, norm weight
        // and bias once, the output written (and read too when accumulating)
        double bytes = 0;
        for (int i = 0; i < g.nseg; ++i) {
            const DevMatrix &W = g.seg[i].W;
            bytes += (double)W.row_bytes * W.N + (W.scales ? (double)W.N * (W.K / 32) * 2 : 0.0);
            if (!g.gate_up || i == 0) bytes += (double)g.rows * W.N * 4 * (g.seg[i].epi == EPI_ADD ? 2 : 1);
            if (g.seg[i].bias) bytes += (double)W.N * 4;
        }
        bytes += (double)g.rows * g.seg[0].W.K * 4 + (g.norm_w ? g.seg[0].W.K * 4.0 : 0.0);
        if (pre.t) bytes += 3.0 * g.seg[0].W.K * 4;   // t, its norm weight, x_new written
        if (g.rows == 1) {
            Node nd = pre.t ? make_node(what + " with the post-branch norm", 1, [g, sms, pre](cudaStream_t s) { launch_gemv(g, sms, s, &pre); })
                            : make_node(what, 1, [g, sms](cudaStream_t s) { launch_gemv(g, sms, s); });
            nd.kind = "gemv";
            nd.bytes = [bytes](int) { return bytes; };
            P.nodes.push_back(nd);
        } else {
            // bulk rows: the prologue norm and the gated form are not fused on this path
            if (g.norm_w || g.gate_up) throw Error{SYN_E_UNSUPPORTED_OP, "internal: fused bulk matmul"};
            double flops = 0;
            for (int i = 0; i < g.nseg; ++i) flops += 2.0 * g.rows * g.seg[i].W.N * g.seg[i].W.K;
            if (opt_tc && gemm_tc_supported(g)) {
                auto sc = c.tc;
                sc->x_bytes = std::max(sc->x_bytes, gemm_tc_x_bytes(g));
                sc->w_bytes = std::max(sc->w_bytes, gemm_tc_w_bytes(g));
                int *err = &d_state->err;
                // resident operand planes of each segment's weight, if built
                std::array<const void *, 3> planes = {nullptr, nullptr, nullptr};
                int launches = 1 + g.nseg;
                for (int i = 0; i < g.nseg; ++i) {
                    auto it = plane_of.find(g.seg[i].W.codes);
                    if (it != plane_of.end()) planes[i] = it->second;
                    launches += planes[i] ? 0 : 1;
                }
                Node nd = make_node(what, launches, [g, planes, sc, err](cudaStream_t s) {
                    CUDA_TRY(launch_gemm_tc(g, planes.data(), sc->x, sc->w, err, s));
                });
                nd.kind = "gemm_tc";
                nd.bytes = [bytes](int) { return bytes; };
                nd.flops = flops;
                P.nodes.push_back(nd);
            } else {
                Node nd = make_node(what, g.nseg, [g](cudaStream_t s) { launch_gemm_rows(g, s); });
                nd.kind = "gemm";
                nd.bytes = [bytes](int) { return bytes; };
                nd.flops = flops;
                P.nodes.push_back(nd);
            }
        }
    }

    // one archdef step, unfused
    void emit_single(Plan &P, Ctx &c, const Step &st, int layer) {
        const std::string &op = st.op;
        const std::string where = op + " (line " + std::to_string(st.line) + (layer >= 0 ? ", layer " + std::to_string(layer) : "") + ")";
        auto src_buf = [&](int i) { return c.buf.at(st.args[i]); };
        float *dst = c.buf.at(st.dst);
        const int rows = op == "embed" ? c.n : c.rows.at(st.args[0]);
        if (op == "embed") {
            EmbedParams e;
            e.E = tensor(st, 0, layer).mat;
            e.tokens = d_tokens;
            e.n = c.n;
            e.out = dst;
            e.state = d_state;
            Node nd = make_node(where, 1, [e](cudaStream_t s) { launch_embed(e, s); });
            P.nodes.push_back(nd);
        } else if (op == "rms_norm") {
            RmsParams r;
            r.x = src_buf(0);
            r.y = dst;
            r.w = tensor(st, 1, layer).vec();
            r.rows = rows;
            r.width = (int)tensor(st, 1, layer).ne[0];
            r.ld = ld(st.args[0]);
            r.eps = eps;
            if (ld(st.args[0]) != ld(st.dst)) throw Error{SYN_E_UNSUPPORTED_OP, "rms_norm between registers of different widths"};
            Node nd = make_node(where, 1, [r](cudaStream_t s) { launch_rmsnorm(r, s); });
            P.nodes.push_back(nd);
        } else if (op == "matmul") {
            const DevTensor &t = tensor(st, 1, layer);
            float *out = dst;
            bool alias = st.dst == st.args[0];
            if (alias) out = c.tmp;
            emit_matmul(P, c, {seg_for(t, out, st.dst)}, st.args[0], 0, where);
            if (alias) {
                float *d = dst;
                const float *tmp = c.tmp;
                size_t bytes = (size_t)rows * ld(st.dst) * sizeof(float);
                Node nd = make_node(where + " copy", 0, [d, tmp, bytes](cudaStream_t s) {
                    cudaMemcpyAsync(d, tmp, bytes, cudaMemcpyDeviceToDevice, s);
                });
                P.nodes.push_back(nd);
            }
        } else if (op == "add_bias" || is_act(op) || op == "mul" || op == "add" || op == "scale" || op == "copy") {
            EltParams e;
            e.y = dst;
            e.a = src_buf(0);
            e.rows = rows;
            e.width = reg_width.at(st.args[0]);
            e.ld = ld(st.args[0]);
            if (ld(st.args[0]) != ld(st.dst)) throw Error{SYN_E_UNSUPPORTED_OP, where + ": registers of different widths"};
            if (op == "add_bias") { e.op = ELT_BIAS; e.b = tensor(st, 1, layer).vec(); }
            else if (is_act(op)) { e.op = ELT_ACT; e.act = act_code(op); }
            else if (op == "mul") { e.op = ELT_MUL; e.b = src_buf(1); }
            else if (op == "add") { e.op = ELT_ADD; e.b = src_buf(1); }
            else if (op == "scale") { e.op = ELT_SCALE; e.c = scale_value(st.args[1]); }
            else e.op = ELT_COPY;
            Node nd = make_node(where, 1, [e](cudaStream_t s) { launch_eltwise(e, s); });
            P.nodes.push_back(nd);
        } else if (op == "norm_heads" || op == "rope") {
            HeadsParams h;
            if (st.dst != st.args[0]) {
                // assignment form: copy, then transform in place
                float *d = dst;
                const float *sbuf = src_buf(0);
                size_t bytes = (size_t)rows * ld(st.dst) * sizeof(float);
                Node nd = make_node(where + " copy", 0, [d, sbuf, bytes](cudaStream_t s) {
                    cudaMemcpyAsync(d, sbuf, bytes, cudaMemcpyDeviceToDevice, s);
                });
                P.nodes.push_back(nd);
            }
            h.q = dst;
            h.ldq = ld(st.dst);
            h.hd = head_dim;
            h.rows = rows;
            h.eps = eps;
            h.state = d_state;
            h.rope_cs = rope_cs;
            h.rope_adjacent = ad.rope_adjacent;
            if (op == "norm_heads") {
                h.nq = head_count(st.args[2]);
                h.wq = tensor(st, 1, layer).vec();
            } else {
                h.nq = head_count(st.args[1]);
                h.rope_q = 1;
            }
            Node nd = make_node(where, 1, [h](cudaStream_t s) { launch_heads(h, s); });
            P.nodes.push_back(nd);
        } else if (op == "attention") {
            emit_attention(P, c, st, layer, nullptr);
        } else if (op == "last") {
            // keep the last row: row n-1 moves to row 0
            float *d = dst;
            const float *sbuf = src_buf(0);
            int w = (int)ld(st.dst);
            if (rows > 1 || d != sbuf) {
                const float *from = sbuf + (size_t)(rows - 1) * ld(st.args[0]);
                Node nd = make_node(where, 0, [d, from, w](cudaStream_t s) { launch_copy_row(d, from, w, s); });
                P.nodes.push_back(nd);
            }
            c.rows[st.dst] = 1;
            return;
        } else {
            throw Error{SYN_E_UNSUPPORTED_OP, "op " + op + " is not implemented"};
        }
        c.rows[st.dst] = rows;
    }

    // attention (+ the q/k transforms and KV append that precede it when `prep` is given)
    struct Prep {
        const float *wq = nullptr, *wk = nullptr;
        int rope_q = 0, rope_k = 0;
    };
    void emit_attention(Plan &P, Ctx &c, const Step &st, int layer, const Prep *prep) {
        const int rows = c.rows.at(st.args[0]);
        HeadsParams h;
        h.hd = head_dim;
        h.rows = rows;
        h.eps = eps;
        h.state = d_state;
        h.rope_cs = rope_cs;
        h.rope_adjacent = ad.rope_adjacent;
        h.k = c.buf.at(st.args[1]);
        h.ldk = ld(st.args[1]);
        h.nk = n_head_kv;
        h.v = c.buf.at(st.args[2]);
        h.ldv = ld(st.args[2]);
        const size_t layer_off = (size_t)layer * n_head_kv * max_ctx * head_dim * kv_es;
        h.kcache = static_cast<uint8_t *>(kcache) + layer_off;
        h.vcache = static_cast<uint8_t *>(vcache) + layer_off;
        h.max_ctx = max_ctx;
        h.kv_f16 = kv_es == 2;
        if (prep) {
            h.q = c.buf.at(st.args[0]);
            h.ldq = ld(st.args[0]);
            h.nq = n_head;
            h.wq = prep->wq;
            h.wk = prep->wk;
            h.rope_q = prep->rope_q;
            h.rope_k = prep->rope_k;
        }
        const std::string where = "attention (line " + std::to_string(st.line) + ", layer " + std::to_string(layer) + ")";
        // decode with the fusion pass: the per-head transforms and the KV append run inside the
        // attention kernel
        const bool fold_heads = prep && rows == 1 && c.fused;
        if (!fold_heads) {
            Node nd = make_node(where + " kv-append", 1, [h](cudaStream_t s) { launch_heads(h, s); });
            nd.kind = "heads";
            const double hb = (double)rows * ((prep ? 2.0 * n_head : 0.0) + 4.0 * n_head_kv) * head_dim * 4;
            nd.bytes = [hb](int) { return hb; };
            P.nodes.push_back(nd);
        }
        AttnParams a;
        a.q = c.buf.at(st.args[0]);
        a.ldq = ld(st.args[0]);
        a.out = c.buf.at(st.dst);
        a.ldo = ld(st.dst);
        a.kcache = static_cast<const uint8_t *>(kcache) + layer_off;
        a.vcache = static_cast<const uint8_t *>(vcache) + layer_off;
        a.kv_f16 = kv_es == 2;
        a.n_head = n_head;
        a.n_kv = n_head_kv;
        a.hd = head_dim;
        a.max_ctx = max_ctx;
        a.rows = rows;
        a.window = layer_windowed(layer) ? window : 0;
        a.splits = c.splits;
        a.part = c.part;
        a.counters = attn_counters;
        a.state = d_state;
        a.err = &d_state->err;
        if (fold_heads) {
            a.fuse_heads = 1;
            a.heads = h;
        }
        if (rows > 1 && opt_attn_tc && attention_tc_supported(a)) {
            // bulk prefill on the tensor cores: split q and the cache into f16 hi/lo planes, then
            // S = Q K^T and O = P V per query head and 128-row block
            auto sc = c.atc;
            sc->q_bytes = std::max(sc->q_bytes, attention_tc_q_bytes(a));
            sc->kv_bytes = std::max(sc->kv_bytes, attention_tc_kv_bytes(a));
            Node nd = make_node(where, 3, [a, sc](cudaStream_t s) { CUDA_TRY(launch_attention_tc(a, sc->q, sc->kv, s)); });
            nd.kind = "attention_tc";
            const int kvh = n_head_kv, hd = head_dim, win = a.window, nr = rows, nh = n_head;
            const size_t es = kv_es;
            // bytes: the cache prefix once (the tiles are shared through L2), q in and the output out
            nd.bytes = [kvh, hd, nr, nh, es](int pos) {
                return 2.0 * kvh * hd * (double)es * (pos + nr) + 2.0 * nr * nh * hd * 4.0;
            };
            // f32-equivalent flops of S and P V over the allowed keys of every row and head
            nd.flops_at = [hd, win, nr, nh](int pos) {
                double keys = 0;
                for (int r = 0; r < nr; ++r) {
                    const int p = pos + r;
                    keys += win > 0 ? std::min(p + 1, win) : p + 1;
                }
                return 4.0 * nh * hd * keys;
            };
            P.nodes.push_back(nd);
        } else {
            Node nd = make_node(where, 1, [a](cudaStream_t s) { launch_attention(a, s); });
            nd.kind = "attention";
            // K and V of every allowed key once, per row; q in, a out
            const int kvh = n_head_kv, hd = head_dim, win = a.window, nr = rows, nh = n_head;
            const size_t es = kv_es;
            nd.bytes = [kvh, hd, win, nr, nh, es](int pos) {
                double b = 0;
                for (int r = 0; r < nr; ++r) {
                    const int p = pos + r;
                    const int len = win > 0 ? std::min(p + 1, win) : p + 1;
                    b += 2.0 * kvh * hd * (double)es * len + 2.0 * nh * hd * 4.0;
                }
                return b;
            };
            P.nodes.push_back(nd);
        }
        c.rows[st.dst] = rows;
    }

    // Try the fusion patterns at step i; returns the number of steps consumed (0 = no match).
    size_t try_fuse(Plan &P, Ctx &c, int sec, size_t i, int layer) {
        const auto &S = ad.sec[sec];
        const Step &st = S[i];
        auto at = [&](size_t j) -> const Step * { return j < S.size() ? &S[j] : nullptr; };

        // (1) `h = rms_norm(x, w)` read only by matmuls (and `last`) before h is overwritten, with x
        //     unchanged meanwhile: normalise inside the matmuls' prologue, never materialise h.
        if (st.op == "rms_norm" && c.rows.at(st.args[0]) == 1) {
            const std::string h = st.dst, x = st.args[0];
            bool ok = true, any = false;
            // the steps that follow, in execution order (a block wraps to the next layer's start,
            // where the block reassigns h before reading it again)
            std::vector<const Step *> seq;
            for (size_t j = i + 1; j < S.size(); ++j) seq.push_back(&S[j]);
            if (sec == 1)
                for (size_t j = 0; j <= i; ++j) seq.push_back(&S[j]);
            if (sec == 0)
                for (auto &s2 : ad.sec[1]) seq.push_back(&s2);
            bool x_written = false;
            for (const Step *s2 : seq) {
                if (reads(*s2, h)) {
                    if (!(s2->op == "matmul" || (s2->op == "last" && s2->dst == h)) || x_written) { ok = false; break; }
                    if (s2->op == "matmul") any = true;
                    if (s2->op == "matmul" && s2->dst == h) break;
                }
                if (s2->assign && s2->dst == h && !reads(*s2, h)) break;
                if (s2->dst == x && h != x) x_written = true;
            }
            if (ok && any && h != x) {
                c.fold_rms[h] = {x, tensor(st, 1, layer).vec()};
                c.rows[h] = 1;
                P.folded.insert(h);
                return 1;
            }
            if (ok && any && h == x) {
                // in-place epilogue norm: x = rms_norm(x, w); [x = last(x)]; y = matmul(x, W)
                // keep the pre-norm values in x (last is row-wise, so it commutes with the norm)
                c.fold_rms[h] = {x, tensor(st, 1, layer).vec()};
                P.folded.insert(h + " (normalised)");
                return 1;
            }
        }

        // (2) the gated feed-forward: g = matmul(h, Wg); act(g); u = matmul(h, Wu); mul(g, u)
        //     (the act may also come after the second matmul), u dead afterwards.
        if (st.op == "matmul") {
            const Step *a1 = at(i + 1), *a2 = at(i + 2), *a3 = at(i + 3);
            const Step *act = nullptr, *mm2 = nullptr, *mul = nullptr;
            if (a1 && a2 && a3) {
                if (is_act(a1->op) && !a1->assign && a1->dst == st.dst && a2->op == "matmul") { act = a1; mm2 = a2; }
                else if (a1->op == "matmul" && is_act(a2->op) && !a2->assign && a2->dst == st.dst) { mm2 = a1; act = a2; }
                mul = a3;
            }
            if (act && mm2 && mul && mm2->args[0] == st.args[0] && mm2->dst != st.dst && mm2->dst != st.args[0] &&
                mul->op == "mul" && !mul->assign && mul->args[0] == st.dst && mul->args[1] == mm2->dst &&
                dead_after(mm2->dst, sec, i + 3) && st.dst != st.args[0]) {
                const DevTensor &wg = tensor(st, 1, layer), &wu = tensor(*mm2, 1, layer);
                const int rows = c.rows.at(st.args[0]);
                if (rows > 1 && wg.mat.N == wu.mat.N) {
                    // bulk rows: the two matmuls on one split of their shared input, then
                    // g = act(g) * u in one elementwise pass
                    if (wg.mat.K == wu.mat.K) {
                        emit_matmul(P, c, {seg_for(wg, c.buf.at(st.dst), st.dst), seg_for(wu, c.buf.at(mm2->dst), mm2->dst)}, st.args[0], 0,
                                    "gate+up matmuls (line " + std::to_string(st.line) + ", layer " + std::to_string(layer) + ")");
                    } else {
                        emit_matmul(P, c, {seg_for(wg, c.buf.at(st.dst), st.dst)}, st.args[0], 0,
                                    "matmul (line " + std::to_string(st.line) + ", layer " + std::to_string(layer) + ")");
                        emit_matmul(P, c, {seg_for(wu, c.buf.at(mm2->dst), mm2->dst)}, st.args[0], 0,
                                    "matmul (line " + std::to_string(mm2->line) + ", layer " + std::to_string(layer) + ")");
                    }
                    EltParams e;
                    e.y = c.buf.at(st.dst);
                    e.a = c.buf.at(st.dst);
                    e.b = c.buf.at(mm2->dst);
                    e.rows = rows;
                    e.width = (int)wg.mat.N;
                    e.ld = ld(st.dst);
                    e.op = ELT_ACT_MUL;
                    e.act = act_code(act->op);
                    Node nd = make_node(act->op + "*mul (line " + std::to_string(act->line) + ", layer " + std::to_string(layer) + ")", 1,
                                        [e](cudaStream_t s) { launch_eltwise(e, s); });
                    nd.kind = "eltwise";
                    const double eb = 3.0 * rows * (double)wg.mat.N * 4;
                    nd.bytes = [eb](int) { return eb; };
                    P.nodes.push_back(nd);
                    c.rows[st.dst] = rows;
                    c.rows[mm2->dst] = rows;
                    return 4;
                }
                if (rows == 1 && wg.mat.wtype == wu.mat.wtype && wg.mat.K == wu.mat.K && wg.mat.N == wu.mat.N) {
                    GemvSeg g = seg_for(wg, c.buf.at(st.dst), st.dst), u = seg_for(wu, nullptr, mm2->dst);
                    emit_matmul(P, c, {g, u}, st.args[0], act_code(act->op),
                                "gate/up/" + act->op + "/mul (line " + std::to_string(st.line) + ", layer " + std::to_string(layer) + ")");
                    c.rows[st.dst] = 1;
                    P.folded.insert(mm2->dst);
                    return 4;
                }
            }
        }

        // (3) matmuls sharing one input (fused Q/K/V), each optionally followed by its add_bias;
        //     a single matmul followed by `add(x, o)` with o dead afterwards accumulates into x.
        if (st.op == "matmul" && st.dst != st.args[0]) {
            const int rows = c.rows.at(st.args[0]);
            std::vector<GemvSeg> segs;
            std::vector<std::string> outs;
            size_t j = i;
            const DevTensor &t0 = tensor(st, 1, layer);
            while (j < S.size() && segs.size() < 3) {
                const Step &m = S[j];
                if (m.op != "matmul" || m.args[0] != st.args[0] || m.dst == st.args[0]) break;
                if (std::find(outs.begin(), outs.end(), m.dst) != outs.end()) break;
                const DevTensor &t = tensor(m, 1, layer);
                if (t.mat.wtype != t0.mat.wtype || t.mat.K != t0.mat.K) break;
                GemvSeg sg = seg_for(t, c.buf.at(m.dst), m.dst);
                ++j;
                if (j < S.size() && S[j].op == "add_bias" && !S[j].assign && S[j].dst == m.dst) {
                    sg.bias = tensor(S[j], 1, layer).vec();
                    ++j;
                }
                segs.push_back(sg);
                outs.push_back(m.dst);
            }
            if (segs.size() == 1 && j < S.size()) {
                const Step &ad2 = S[j];
                if (ad2.op == "add" && !ad2.assign && ad2.args[1] == outs[0] && ad2.dst != outs[0] &&
                    ad2.dst != st.args[0] && dead_after(outs[0], sec, j) && c.rows.at(ad2.dst) == rows) {
                    segs[0].out = c.buf.at(ad2.dst);
                    segs[0].ldo = ld(ad2.dst);
                    segs[0].epi = EPI_ADD;
                    emit_matmul(P, c, segs, st.args[0], 0,
                                "matmul+residual (line " + std::to_string(st.line) + ", layer " + std::to_string(layer) + ")");
                    P.folded.insert(outs[0]);
                    return j + 1 - i;
                }
            }
            if (segs.size() >= 2 || (segs.size() == 1 && segs[0].bias)) {
                emit_matmul(P, c, segs, st.args[0], 0,
                            "matmul x" + std::to_string(segs.size()) + " (line " + std::to_string(st.line) + ", layer " + std::to_string(layer) + ")");
                for (auto &o : outs) c.rows[o] = rows;
                return j - i;
            }
        }

        // (4) the per-head transforms before attention: norm_heads / rope on q and k (in that
        //     order per register), then a = attention(q, k, v): one kernel transforms q and k and
        //     appends k and v to the cache, then the attention kernel reads the cache.
        if ((st.op == "norm_heads" || st.op == "rope") && !st.assign) {
            Prep pr;
            size_t j = i;
            std::string qn, kn;
            int stage_q = 0, stage_k = 0;  // 0 none, 1 normed, 2 roped
            std::vector<std::pair<std::string, const Step *>> seen;
            while (j < S.size() && (S[j].op == "norm_heads" || S[j].op == "rope") && !S[j].assign) {
                seen.push_back({S[j].dst, &S[j]});
                ++j;
            }
            const Step *att = j < S.size() ? &S[j] : nullptr;
            if (att && att->op == "attention") {
                qn = att->args[0];
                kn = att->args[1];
                bool ok = qn != kn;
                for (auto &pr2 : seen) {
                    const Step &s2 = *pr2.second;
                    int &stage = s2.dst == qn ? stage_q : stage_k;
                    if (s2.dst != qn && s2.dst != kn) { ok = false; break; }
                    if (s2.op == "norm_heads") {
                        if (stage != 0) { ok = false; break; }
                        stage = 1;
                        (s2.dst == qn ? pr.wq : pr.wk) = tensor(s2, 1, layer).vec();
                        int cnt = head_count(s2.args[2]);
                        if (cnt != (s2.dst == qn ? n_head : n_head_kv)) { ok = false; break; }
                    } else {
                        if (stage == 2) { ok = false; break; }
                        stage = 2;
                        (s2.dst == qn ? pr.rope_q : pr.rope_k) = 1;
                        int cnt = head_count(s2.args[1]);
                        if (cnt != (s2.dst == qn ? n_head : n_head_kv)) { ok = false; break; }
                    }
                }
                if (ok && dead_after(kn, sec, j)) {
                    emit_attention(P, c, *att, layer, &pr);
                    P.folded.insert(kn + " (post-rope)");
                    return j + 1 - i;
                }
            }
        }

        // (5) post-branch norm: o = rms_norm(o, w); add(x, o), o dead afterwards -> x += norm(o) w.
        //     In decode, when the next step normalises x for matmuls (`h = rms_norm(x, w2)`, in
        //     this section or at the start of the next layer's block), the update waits for the
        //     first matmul that reads x and runs in its prologue; anything else that touches x
        //     first gets this node in its original place (emit_section).
        if (st.op == "rms_norm" && st.dst == st.args[0]) {
            const Step *a1 = at(i + 1);
            if (a1 && a1->op == "add" && !a1->assign && a1->args[1] == st.dst && a1->dst != st.dst &&
                dead_after(st.dst, sec, i + 1) && ld(a1->dst) == ld(st.dst)) {
                RmsParams r;
                r.x = c.buf.at(st.dst);
                r.w = tensor(st, 1, layer).vec();
                r.rows = c.rows.at(st.dst);
                r.width = (int)ld(st.dst);
                r.ld = ld(st.dst);
                r.eps = eps;
                r.residual = c.buf.at(a1->dst);
                Node nd = make_node("rms_norm+residual (line " + std::to_string(st.line) + ", layer " + std::to_string(layer) + ")", 1,
                                    [r](cudaStream_t s) { launch_rmsnorm(r, s); });
                const Step *nx = at(i + 2);
                if (!nx && sec == 1 && layer + 1 < n_layer) nx = &S[0];
                const std::string x = a1->dst;
                if (r.rows == 1 && r.width % 4 == 0 && nx && nx->op == "rms_norm" && nx->args[0] == x && nx->dst != x &&
                    !c.pre.count(x)) {
                    Ctx::PendingPre pp;
                    pp.t = r.x;
                    pp.w = r.w;
                    pp.at = P.nodes.size();
                    pp.node = nd;
                    c.pre[x] = pp;
                    P.folded.insert(st.dst + " (post-branch norm in the next matmul)");
                    return 2;
                }
                P.nodes.push_back(nd);
                return 2;
            }
        }

        // (6) `x = embed(T)` then `scale(x, c)`: scale inside the gather
        if (st.op == "embed") {
            const Step *a1 = at(i + 1);
            EmbedParams e;
            e.E = tensor(st, 0, layer).mat;
            e.tokens = d_tokens;
            e.n = c.n;
            e.out = c.buf.at(st.dst);
            e.state = d_state;
            size_t used = 1;
            if (a1 && a1->op == "scale" && !a1->assign && a1->dst == st.dst) {
                e.scale = scale_value(a1->args[1]);
                used = 2;
            }
            if (used == 2) {
                Node nd = make_node("embed+scale", 1, [e](cudaStream_t s) { launch_embed(e, s); });
                P.nodes.push_back(nd);
                c.rows[st.dst] = c.n;
                return used;
            }
        }
        return 0;
    }

    // put a pending post-branch update's own node back where it was due
    void flush_pre(Plan &P, Ctx &c, const std::string &x) {
        auto it = c.pre.find(x);
        if (it == c.pre.end()) return;
        const size_t at = it->second.at;
        P.nodes.insert(P.nodes.begin() + (std::ptrdiff_t)at, it->second.node);
        c.pre.erase(it);
        for (auto &o : c.pre)
            if (o.second.at >= at) ++o.second.at;
    }

    void emit_section(Plan &P, Ctx &c, int sec, int layer) {
        const auto &S = ad.sec[sec];
        for (size_t i = 0; i < S.size();) {
            // a pending post-branch update of x: `h = rms_norm(x, w2)` folded into matmuls keeps it
            // waiting (the matmuls take it); any other step that touches x gets the update first
            if (!c.pre.empty()) {
                const Step &st0 = S[i];
                std::vector<std::string> touched;
                for (auto &pp : c.pre)
                    if (reads(st0, pp.first) || st0.dst == pp.first) touched.push_back(pp.first);
                std::string fold_x;   // the register this step may normalise for matmuls
                for (auto &x : touched) {
                    if (c.fused && st0.op == "rms_norm" && st0.args[0] == x && st0.dst != x) fold_x = x;
                    else flush_pre(P, c, x);
                }
                if (!fold_x.empty()) {
                    if (try_fuse(P, c, sec, i, layer) == 1) {   // pattern (1): h is normalised inside the matmuls that read it
                        any_fused = true;
                        ++i;
                        continue;
                    }
                    flush_pre(P, c, fold_x);   // nothing was emitted: the step runs as it is, after the update
                }
            }
            size_t used = c.fused ? try_fuse(P, c, sec, i, layer) : 0;
            if (used) {
                any_fused = true;
                i += used;
                continue;
            }
            const Step &st = S[i];
            // a register whose rms_norm was folded but is read by something the fold did not plan
            if (c.fold_rms.count(st.dst) && st.assign && !reads(st, st.dst)) c.fold_rms.erase(st.dst);
            for (auto &r : reads_of(st))
                if (c.fold_rms.count(r) && st.op != "matmul" && !(st.op == "last" && st.dst == r))
                    throw Error{SYN_E_UNSUPPORTED_OP, "internal: folded register " + r + " read by " + st.op};
            if (st.op == "matmul" && st.dst == st.args[0]) {
                emit_single(P, c, st, layer);
            } else if (st.op == "matmul") {
                const DevTensor &t = tensor(st, 1, layer);
                float *out = c.buf.at(st.dst);
                emit_matmul(P, c, {seg_for(t, out, st.dst)}, st.args[0], 0,
                            "matmul (line " + std::to_string(st.line) + (layer >= 0 ? ", layer " + std::to_string(layer) : "") + ")");
                c.rows[st.dst] = c.rows.at(st.args[0]);
                if (c.fold_rms.count(st.dst)) c.fold_rms.erase(st.dst);
            } else if (st.op == "last" && c.fold_rms.count(st.args[0])) {
                // the folded norm stays attached through the row selection
                auto f = c.fold_rms[st.args[0]];
                emit_single(P, c, st, layer);
                f.first = st.dst;
                c.fold_rms[st.dst] = f;
            } else {
                emit_single(P, c, st, layer);
            }
            ++i;
        }
    }

    Plan &build_plan(Plan &P, int n, bool fused) {
        P.drop_graph();
        P.capture_failed = false;
        P.nodes.clear();
        P.regs.clear();
        P.folded.clear();
        P.n = n;
        P.fused = fused;
        pool.reset();
        Ctx c;
        c.n = n;
        c.fused = fused;   // bulk plans take the patterns that hold for many rows
        for (auto &rw : reg_width) {  // std::map: deterministic order
            const int rows = reg_multi.at(rw.first) ? n : 1;
            c.buf[rw.first] = static_cast<float *>(pool.alloc((size_t)rows * rw.second * sizeof(float)));
            c.rows[rw.first] = rows;
            P.regs[rw.first] = c.buf[rw.first];
        }
        int maxw = 0;
        for (auto &rw : reg_width) maxw = std::max(maxw, rw.second);
        c.tmp = static_cast<float *>(pool.alloc((size_t)n * maxw * sizeof(float)));
        // one attention CTA per SM (each holds a 192 KB copy ring): KV heads x rows x splits <= SMs,
        // the split count the largest power of two that allows (on llama-3-8B decode at 8192 keys,
        // 16 slices per KV head ran about 1 % faster than 19, 17, 15 or 14)
        int pow2 = 1;
        while (pow2 < 64 && (int64_t)2 * pow2 * n_head_kv * n <= sm_count) pow2 *= 2;
        c.splits = opt_splits > 0 ? opt_splits : pow2;
        c.part = static_cast<float *>(pool.alloc((size_t)n * n_head * std::max(c.splits, n == 1 ? 64 : 1) * (head_dim + 4) * sizeof(float)));
        emit_section(P, c, 0, -1);
        for (int l = 0; l < n_layer; ++l) emit_section(P, c, 1, l);
        emit_section(P, c, 2, -1);
        while (!c.pre.empty()) flush_pre(P, c, c.pre.begin()->first);   // no matmul took it
        if (c.tc->x_bytes) {
            c.tc->x = pool.alloc(c.tc->x_bytes);
            c.tc->w = pool.alloc(c.tc->w_bytes);
        }
        if (c.atc->q_bytes) {
            c.atc->q = pool.alloc(c.atc->q_bytes);
            c.atc->kv = pool.alloc(c.atc->kv_bytes);
        }
        ArgmaxParams a;
        a.x = c.buf.at("logits");
        a.n = n_vocab;
        a.part_v = arg_v;
        a.part_i = arg_i;
        a.counter = arg_counter;
        a.state = d_state;
        a.advance = 1;
        const int blocks = arg_blocks;
        {
            Node nd = make_node("argmax+advance", 1, [a, blocks](cudaStream_t s) { launch_argmax(a, blocks, s); });
            P.nodes.push_back(nd);
        }
        // profile categories of the small nodes, from what they do
        for (auto &nd : P.nodes) {
            if (nd.kind != "other") continue;
            const std::string &w = nd.what;
            nd.kind = w.find("copy") != std::string::npos || w.rfind("last", 0) == 0 ? "copy"
                    : w.rfind("embed", 0) == 0 ? "embed"
                    : w.rfind("rms_norm", 0) == 0 ? "rmsnorm"
                    : w.rfind("argmax", 0) == 0 ? "argmax"
                    : (w.rfind("norm_heads", 0) == 0 || w.rfind("rope", 0) == 0) ? "heads" : "eltwise";
        }
        return P;
    }

    void run_plan(const Plan &P) {
        if (!opt_profile) {
            for (auto &nd : P.nodes) nd.run(stream);
            CUDA_TRY(cudaGetLastError());
            return;
        }
        // profile: one event pair around every node, device time accumulated per kind
        while (prof_ev.size() < 2 * P.nodes.size()) {
            cudaEvent_t e;
            CUDA_TRY(cudaEventCreate(&e));
            prof_ev.push_back(e);
        }
        for (size_t i = 0; i < P.nodes.size(); ++i) {
            CUDA_TRY(cudaEventRecord(prof_ev[2 * i], stream));
            P.nodes[i].run(stream);
            CUDA_TRY(cudaEventRecord(prof_ev[2 * i + 1], stream));
        }
        CUDA_TRY(cudaGetLastError());
        CUDA_TRY(cudaStreamSynchronize(stream));
        for (size_t i = 0; i < P.nodes.size(); ++i) {
            float ms = 0.f;
            CUDA_TRY(cudaEventElapsedTime(&ms, prof_ev[2 * i], prof_ev[2 * i + 1]));
            ProfEntry &e = prof[P.nodes[i].kind];
            e.launches += P.nodes[i].launches;
            e.ms += ms;
            if (P.nodes[i].bytes) e.bytes += P.nodes[i].bytes(prof_pos);
            e.flops += P.nodes[i].flops + (P.nodes[i].flops_at ? P.nodes[i].flops_at(prof_pos) : 0.0);
        }
    }
    int prof_pos = 0;  // position of row 0 of the forward being profiled

};

// =============================================================================================
namespace {

syn_status fail(syn_model *m, const Error &e) {
    if (m) m->err = e.msg;
    return e.code;
}

template <class F> syn_status guarded(syn_model *m, F &&f) {
    if (!m) return SYN_E_INVALID_ARG;
    try {
        f();
        m->err.clear();
        return SYN_OK;
    } catch (const Error &e) {
        return fail(m, e);
    } catch (const std::bad_alloc &) {
        return fail(m, Error{SYN_E_OOM, "host allocation failed"});
    } catch (const std::exception &e) {
        return fail(m, Error{SYN_E_STATE, e.what()});
    }
}

size_t round32(size_t b) { return (b + 31) / 32 * 32; }

uint16_t f32_bits_to_half_bits(float f) { return __half_as_ushort(__float2half_rn(f)); }

}  // namespace

// =============================================================================================
// C ABI
// =============================================================================================
extern "C" {

syn_status syn_archdef_check(const char *file_arch, const char *text, size_t len, int *steps_per_layer, char *err,
                             size_t errlen) {
    if (!text) return SYN_E_INVALID_ARG;
    Archdef ad;
    std::string e;
    bool ok = parse_archdef(file_arch ? file_arch : "", std::string(text, len), ad, e);
    if (err && errlen) {
        std::snprintf(err, errlen, "%s", ok ? "" : e.c_str());
    }
    if (ok && steps_per_layer) *steps_per_layer = (int)ad.sec[1].size();
    return ok ? SYN_OK : SYN_E_ARCHDEF;
}

syn_status syn_archdef_sha256(const char *text, size_t len, char *hex65) {
    if ((!text && len) || !hex65) return SYN_E_INVALID_ARG;
    const std::string h = sha256_hex(text ? text : "", len);
    std::memcpy(hex65, h.c_str(), 65);
    return SYN_OK;
}

syn_status syn_describe(syn_model *m, char *buf, size_t len) {
    return guarded(m, [&] {
        if (!buf || !len) throw Error{SYN_E_INVALID_ARG, "null buffer"};
        std::string o = "arch=" + m->ad.arch + " file=" + m->file_arch + " steps_per_layer=" + std::to_string(m->ad.sec[1].size()) +
                        " prologue_steps=" + std::to_string(m->ad.sec[0].size()) + " epilogue_steps=" + std::to_string(m->ad.sec[2].size()) +
                        " sha256=" + m->archdef_sha + " layers=" + std::to_string(m->n_layer) + " hidden=" + std::to_string(m->n_embd) +
                        " heads=" + std::to_string(m->n_head) + " kv_heads=" + std::to_string(m->n_head_kv) +
                        " head_dim=" + std::to_string(m->head_dim) + " max_ctx=" + std::to_string(m->max_ctx) +
                        " kv=" + (m->opt_kv_f16 ? "f16" : "f32");
        if (m->finalized) {
            std::map<std::string, int> by_type;
            static const char *names[] = {"f32", "f16", "q4_0", "?", "?", "?", "?", "?", "q8_0"};
            for (auto &t : m->tensors) {
                const int d = t.second.dtype;
                by_type[(d >= 0 && d <= 8) ? names[d] : "?"]++;
            }
            std::string w;
            for (auto &b : by_type) w += (w.empty() ? "" : ",") + b.first + ":" + std::to_string(b.second);
            o += " vocab=" + std::to_string(m->n_vocab) + " weights=" + w +
                 " tied=" + (m->tensors.count("output.weight") ? "0" : "1") + " fused=" + (m->any_fused ? "1" : "0") +
                 " kernels_per_step=" + std::to_string(m->decode.launches());
        }
        // the bulk-prefill configuration in effect
        o += std::string(" bulk_matmul=") + (m->opt_tc ? "tc" : "cuda_core") +
             " bulk_attention=" + (m->opt_attn_tc ? "tc" : "ring") + " tc_planes=" +
             (m->opt_tc_planes == 0 ? std::string("off") : m->plane_bytes ? std::to_string(m->plane_bytes)
                                                         : m->opt_tc_planes < 0 ? std::string("auto") : std::string("on"));
        if (o.size() + 1 > len) throw Error{SYN_E_INVALID_ARG, "buffer too small: need " + std::to_string(o.size() + 1)};
        std::memcpy(buf, o.c_str(), o.size() + 1);
    });
}

syn_status syn_create(const char *file_arch, const char *text, size_t len, const char *metadata, int max_ctx,
                      void *cuda_stream, syn_model **out) {
    if (!out || !text || !metadata) return SYN_E_INVALID_ARG;
    *out = nullptr;
    syn_model *m = new (std::nothrow) syn_model();
    if (!m) return SYN_E_OOM;
    *out = m;
    m->t_create = std::chrono::steady_clock::now();
    return guarded(m, [&] {
        m->file_arch = file_arch ? file_arch : "";
        m->archdef_sha = sha256_hex(text, len);
        std::string e;
        if (!parse_archdef(m->file_arch, std::string(text, len), m->ad, e)) throw Error{SYN_E_ARCHDEF, e};
        if (m->file_arch.empty()) m->file_arch = m->ad.arch;
        std::stringstream ms(metadata);
        std::string line;
        while (std::getline(ms, line)) {
            size_t eq = line.find('=');
            if (eq == std::string::npos) continue;
            auto trim = [](std::string s) {
                size_t a = s.find_first_not_of(" \t\r"), b = s.find_last_not_of(" \t\r");
                return a == std::string::npos ? std::string() : s.substr(a, b - a + 1);
            };
            m->meta[trim(line.substr(0, eq))] = trim(line.substr(eq + 1));
        }
        if (max_ctx <= 0) throw Error{SYN_E_INVALID_CONFIG, "max_ctx must be positive"};
        m->max_ctx = max_ctx;
        m->n_layer = m->meta_int("block_count", true);
        m->n_embd = m->meta_int("embedding_length", true);
        m->n_head = m->meta_int("head_count", true);
        m->n_head_kv = m->meta_int("head_count_kv", true);
        m->head_dim = m->meta_int("key_length", false, m->n_head ? m->n_embd / m->n_head : 0);
        m->eps = (float)m->meta_double("layer_norm_rms_epsilon");
        m->rope_base = m->meta_double("freq_base");
        m->window = m->meta_int("sliding_window", false, 0);
        if (m->n_layer <= 0 || m->n_embd <= 0)
            throw Error{SYN_E_INVALID_CONFIG, "block_count and embedding_length must be positive"};
        if (m->n_head <= 0 || m->n_head_kv <= 0 || m->n_head % m->n_head_kv)
            throw Error{SYN_E_INVALID_CONFIG, "head_count must be a positive multiple of head_count_kv"};
        if (m->eps < 0 || m->rope_base <= 0 || m->window < 0)
            throw Error{SYN_E_INVALID_CONFIG, "layer_norm_rms_epsilon must be >= 0, rope.freq_base > 0 and sliding_window >= 0"};
        if (m->head_dim != 64 && m->head_dim != 128 && m->head_dim != 256)
            throw Error{SYN_E_UNSUPPORTED_OP, "head_dim " + std::to_string(m->head_dim) + " (supported: 64, 128, 256)"};
        if (m->n_head / m->n_head_kv > (m->head_dim == 256 ? 4 : 8))
            throw Error{SYN_E_UNSUPPORTED_OP, "too many query heads per KV head (max 8, or 4 with head_dim 256)"};
        // a scale factor is a number or a GGUF metadata key ("Local inference and architectures",
        // section "The operations"); anything else is refused here instead of read as 0
        for (int sec = 0; sec < 3; ++sec)
            for (const Step &st : m->ad.sec[sec]) {
                if (st.op != "scale" || st.args.size() < 2) continue;
                const std::string *mv = m->meta_arch(st.args[1]);
                const std::string &txt = mv ? *mv : st.args[1];
                char *end = nullptr;
                const double c = std::strtod(txt.c_str(), &end);
                if (end == txt.c_str() || *end || !std::isfinite(c))
                    throw Error{SYN_E_ARCHDEF, m->file_arch + ".archdef: line " + std::to_string(st.line) + ": scale factor '" +
                                                   st.args[1] + "' is neither a finite number nor a GGUF metadata key"};
            }
        int ndev = 0;
        if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) throw Error{SYN_E_BACKEND_INIT, "no CUDA device"};
        CUDA_TRY(cudaGetDevice(&m->device));
        cudaDeviceProp prop;
        CUDA_TRY(cudaGetDeviceProperties(&prop, m->device));
        if (prop.major != 10 || prop.minor != 3)
            throw Error{SYN_E_BACKEND_INIT, std::string("device ") + prop.name + " is sm_" + std::to_string(prop.major) +
                                                std::to_string(prop.minor) + "; this library targets sm_103 (GB300)"};
        m->sm_count = prop.multiProcessorCount;
        if (cuda_stream) {
            m->stream = (cudaStream_t)cuda_stream;
        } else {
            CUDA_TRY(cudaStreamCreateWithFlags(&m->stream, cudaStreamNonBlocking));
            m->own_stream = true;
        }
        CUDA_TRY(cudaEventCreate(&m->ev0));
        CUDA_TRY(cudaEventCreate(&m->ev1));
        CUDA_TRY(cudaMallocHost(&m->h_stage, sizeof(int) * syn_model::kStageSlots * syn_model::kStageInts));
        CUDA_TRY(cudaMallocHost(&m->h_out, 2 * sizeof(int)));
        for (auto &e : m->stage_ev) CUDA_TRY(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    });
}

syn_status syn_load_weights(syn_model *m, const char *gguf_name, syn_dtype dtype, const int64_t *ne, int n_dims,
                            const void *host_bytes, size_t nbytes) {
    return guarded(m, [&] {
        if (!gguf_name || !ne || !host_bytes) throw Error{SYN_E_INVALID_ARG, "null argument"};
        if (m->finalized) throw Error{SYN_E_STATE, "syn_load_weights after syn_finalize"};
        const std::string name = gguf_name;
        if (n_dims < 1 || n_dims > 2) throw Error{SYN_E_WEIGHT_FORMAT, name + ": n_dims must be 1 or 2"};
        const int64_t K = ne[0], N = n_dims == 2 ? ne[1] : 1;
        if (K <= 0 || N <= 0) throw Error{SYN_E_WEIGHT_FORMAT, name + ": empty shape"};
        // the kernels index rows and columns with 32-bit integers
        if (K > INT32_MAX || N > INT32_MAX)
            throw Error{SYN_E_WEIGHT_FORMAT, name + ": dimension " + std::to_string(std::max(K, N)) + " is too large (limit 2^31 - 1)"};
        size_t want = 0;
        switch (dtype) {
        case SYN_F32: want = (size_t)K * N * 4; break;
        case SYN_F16: want = (size_t)K * N * 2; break;
        case SYN_Q8_0:
        case SYN_Q4_0:
            if (K % 32) throw Error{SYN_E_WEIGHT_FORMAT, name + ": ne[0]=" + std::to_string(K) + " is not a whole number of 32-weight blocks"};
            want = (size_t)(K / 32) * N * (dtype == SYN_Q8_0 ? 34 : 18);
            break;
        default: throw Error{SYN_E_WEIGHT_FORMAT, name + ": unsupported GGUF type " + std::to_string((int)dtype)};
        }
        if (nbytes != want)
            throw Error{SYN_E_WEIGHT_FORMAT, name + ": declared type " + std::to_string((int)dtype) + " shape needs " +
                                                 std::to_string(want) + " bytes, got " + std::to_string(nbytes)};
        DevTensor t;
        t.name = name;
        t.dtype = dtype;
        t.ne[0] = K;
        t.ne[1] = N;
        t.n_dims = n_dims;
        const uint8_t *src = static_cast<const uint8_t *>(host_bytes);
        std::vector<uint8_t> host;
        size_t codes_bytes = 0, scales_bytes = 0, row_bytes = 0;
        int64_t scale_stride = 0;
        if (n_dims == 1) {
            // vectors (norm weights, biases) are kept as f32
            if (dtype != SYN_F32 && dtype != SYN_F16) throw Error{SYN_E_WEIGHT_FORMAT, name + ": vectors must be f32 or f16"};
            host.resize((size_t)K * 4);
            float *f = reinterpret_cast<float *>(host.data());
            for (int64_t i = 0; i < K; ++i) {
                if (dtype == SYN_F32) std::memcpy(&f[i], src + 4 * i, 4);
                else { uint16_t h; std::memcpy(&h, src + 2 * i, 2); f[i] = __half2float(__ushort_as_half(h)); }
            }
            row_bytes = (size_t)K * 4;
            codes_bytes = host.size();
            t.mat.wtype = W_F32;
        } else if (dtype == SYN_F32 || dtype == SYN_F16) {
            const size_t es = dtype == SYN_F32 ? 4 : 2;
            row_bytes = round32((size_t)K * es);
            codes_bytes = row_bytes * N;
            host.assign(codes_bytes, 0);
            for (int64_t r = 0; r < N; ++r) std::memcpy(host.data() + r * row_bytes, src + (size_t)r * K * es, (size_t)K * es);
            t.mat.wtype = dtype == SYN_F32 ? W_F32 : W_F16;
        } else {
            // split GGUF blocks {f16 d; codes} into a codes array and a scales array; Q8_0 codes
            // become offset-binary (q + 128) so the kernels decode them without a sign fix-up
            const bool q8 = dtype == SYN_Q8_0;
            const size_t blk = q8 ? 34 : 18, cb = q8 ? 32 : 16;
            const int64_t nb = K / 32;
            row_bytes = round32((size_t)nb * cb);
            // one scale per block, padding included, rounded up to 8 scales so that every row's
            // scales start 16-byte aligned
            scale_stride = (int64_t)((row_bytes / cb + 7) / 8 * 8);
            codes_bytes = row_bytes * N;
            scales_bytes = (size_t)scale_stride * N * 2;
            const size_t scales_off = (codes_bytes + 255) / 256 * 256;
            host.assign(scales_off + scales_bytes, 0);
            uint16_t *sc = reinterpret_cast<uint16_t *>(host.data() + scales_off);
            for (int64_t r = 0; r < N; ++r)
                for (int64_t b = 0; b < nb; ++b) {
                    const uint8_t *bp = src + ((size_t)r * nb + b) * blk;
                    std::memcpy(&sc[(size_t)r * scale_stride + b], bp, 2);
                    uint8_t *dst = host.data() + (size_t)r * row_bytes + (size_t)b * cb;
                    if (q8) {
                        for (int j = 0; j < 32; ++j) dst[j] = (uint8_t)(bp[2 + j] ^ 0x80u);
                    } else {
                        std::memcpy(dst, bp + 2, cb);
                    }
                }
            codes_bytes = scales_off;
            t.mat.wtype = q8 ? W_Q8_0 : W_Q4_0;
        }
        t.bytes = host.size();
        cudaError_t e = cudaMalloc(&t.mem, t.bytes);
        if (e != cudaSuccess) throw Error{SYN_E_OOM, name + ": cudaMalloc of " + std::to_string(t.bytes) + " bytes failed"};
        e = cudaMemcpy(t.mem, host.data(), t.bytes, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) {
            cudaFree(t.mem);
            throw Error{SYN_E_CUDA, name + ": upload failed: " + cudaGetErrorString(e)};
        }
        t.mat.K = K;
        t.mat.N = N;
        t.mat.codes = t.mem;
        t.mat.row_bytes = row_bytes;
        t.mat.scale_stride = scale_stride;
        t.mat.scales = scales_bytes ? reinterpret_cast<const uint16_t *>(static_cast<uint8_t *>(t.mem) + codes_bytes) : nullptr;
        auto old = m->tensors.find(name);
        if (old != m->tensors.end()) cudaFree(old->second.mem);
        m->tensors[name] = t;
    });
}

syn_status syn_finalize(syn_model *m) {
    return guarded(m, [&] {
        if (m->finalized) throw Error{SYN_E_STATE, "syn_finalize called twice"};
        m->infer_shapes();
        // every tensor named anywhere must resolve, in every layer
        for (int sec = 0; sec < 3; ++sec)
            for (int l = 0; l < (sec == 1 ? m->n_layer : 1); ++l)
                for (auto &st : m->ad.sec[sec]) {
                    static const std::map<std::string, int> targ = {{"embed", 0}, {"rms_norm", 1}, {"matmul", 1}, {"add_bias", 1}, {"norm_heads", 1}};
                    auto it = targ.find(st.op);
                    if (it == targ.end()) continue;
                    const DevTensor &t = m->tensor(st, it->second, sec == 1 ? l : -1);
                    if ((st.op == "rms_norm" || st.op == "add_bias" || st.op == "norm_heads") && t.n_dims != 1)
                        throw Error{SYN_E_SHAPE_MISMATCH, t.name + " must be a vector for " + st.op};
                }
        m->kv_es = m->opt_kv_f16 ? 2 : 4;
        const size_t kv = (size_t)m->n_layer * m->n_head_kv * m->max_ctx * m->head_dim * m->kv_es;
        cudaError_t e = cudaMalloc(&m->kcache, kv);
        if (e == cudaSuccess) e = cudaMalloc(&m->vcache, kv);
        if (e != cudaSuccess) throw Error{SYN_E_OOM, "KV cache: cudaMalloc of 2 x " + std::to_string(kv) + " bytes failed"};
        CUDA_TRY(cudaMemset(m->kcache, 0, kv));
        CUDA_TRY(cudaMemset(m->vcache, 0, kv));
        // RoPE cos/sin cache ("Execution contract", section "Position caches"): angle p * base^(-2j/hd)
        // evaluated in double, stored as f32 pairs [max_ctx][hd/2]
        const int half = m->head_dim / 2;
        std::vector<float2> cs((size_t)m->max_ctx * half);
        for (int p = 0; p < m->max_ctx; ++p)
            for (int j = 0; j < half; ++j) {
                const double ang = (double)p * std::pow(m->rope_base, -2.0 * j / m->head_dim);
                cs[(size_t)p * half + j] = make_float2((float)std::cos(ang), (float)std::sin(ang));
            }
        CUDA_TRY(cudaMalloc(&m->rope_cs, cs.size() * sizeof(float2)));
        CUDA_TRY(cudaMemcpy(m->rope_cs, cs.data(), cs.size() * sizeof(float2), cudaMemcpyHostToDevice));
        CUDA_TRY(cudaMalloc(&m->d_state, sizeof(DevState)));
        CUDA_TRY(cudaMemset(m->d_state, 0, sizeof(DevState)));
        CUDA_TRY(cudaMalloc(&m->d_tokens, (size_t)m->max_ctx * sizeof(int)));
        m->arg_blocks = std::max(1, std::min(2 * m->sm_count, (m->n_vocab + 4095) / 4096));
        CUDA_TRY(cudaMalloc(&m->arg_v, m->arg_blocks * sizeof(float)));
        CUDA_TRY(cudaMalloc(&m->arg_i, m->arg_blocks * sizeof(int)));
        CUDA_TRY(cudaMalloc(&m->arg_counter, sizeof(unsigned)));
        CUDA_TRY(cudaMemset(m->arg_counter, 0, sizeof(unsigned)));
        CUDA_TRY(cudaMalloc(&m->attn_counters, (size_t)m->max_ctx * m->n_head_kv * sizeof(unsigned)));
        CUDA_TRY(cudaMemset(m->attn_counters, 0, (size_t)m->max_ctx * m->n_head_kv * sizeof(unsigned)));
        m->finalized = true;
        m->tm.load_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - m->t_create).count();
        m->tm.kv_bytes = (int64_t)(2 * kv);
        int64_t wb = 0;
        for (auto &t : m->tensors) wb += (int64_t)t.second.bytes;
        m->tm.weight_bytes = wb;
        // build the decode plan once, so that plan errors surface at load time
        m->build_plan(m->decode, 1, m->opt_fusion != 0);
        m->decode_ready = true;
        m->decode_runs = 0;
    });
}

syn_status syn_reset_kv(syn_model *m) {
    return guarded(m, [&] {
        if (!m->finalized) throw Error{SYN_E_STATE, "syn_reset_kv before syn_finalize"};
        m->kv_len = 0;
    });
}

syn_status syn_forward(syn_model *m, const int32_t *tokens, int n, int pos, float *logits, int32_t *argmax_out,
                       unsigned flags) {
    return guarded(m, [&] {
        if (!m->finalized) throw Error{SYN_E_STATE, "syn_forward before syn_finalize"};
        if (!tokens || n < 1) throw Error{SYN_E_INVALID_ARG, "need at least one token"};
        if (pos != m->kv_len)
            throw Error{SYN_E_STATE, "pos " + std::to_string(pos) + " != KV length " + std::to_string(m->kv_len)};
        if ((int64_t)pos + n > m->max_ctx)
            throw Error{SYN_E_CONTEXT_FULL, "pos + n = " + std::to_string((int64_t)pos + n) + " exceeds max_ctx " + std::to_string(m->max_ctx)};
        cudaStream_t s = m->stream;
        if (!(flags & SYN_TOKENS_ON_DEVICE)) {
            for (int i = 0; i < n; ++i)
                if (tokens[i] < 0 || tokens[i] >= m->n_vocab)
                    throw Error{SYN_E_INVALID_ARG, "token " + std::to_string(tokens[i]) + " at index " + std::to_string(i) +
                                                       " is outside the vocabulary [0, " + std::to_string(m->n_vocab) + ")"};
        }
        const bool dirty = m->dev_pos != pos || m->dev_n != n;
        if ((flags & SYN_TOKENS_ON_DEVICE) || n + 2 > syn_model::kStageInts) {
            CUDA_TRY(cudaMemcpyAsync(m->d_tokens, tokens, (size_t)n * sizeof(int), cudaMemcpyDefault, s));
            if (dirty) {
                int st[2] = {pos, n};
                CUDA_TRY(cudaMemcpyAsync(m->d_state, st, sizeof st, cudaMemcpyHostToDevice, s));
            }
        } else {
            const int slot = m->stage_i;
            m->stage_i = (m->stage_i + 1) % syn_model::kStageSlots;
            CUDA_TRY(cudaEventSynchronize(m->stage_ev[slot]));
            int *h = m->h_stage + slot * syn_model::kStageInts;
            h[0] = pos;
            h[1] = n;
            std::memcpy(h + 2, tokens, (size_t)n * sizeof(int));
            CUDA_TRY(cudaMemcpyAsync(m->d_tokens, h + 2, (size_t)n * sizeof(int), cudaMemcpyHostToDevice, s));
            if (dirty) CUDA_TRY(cudaMemcpyAsync(m->d_state, h, 2 * sizeof(int), cudaMemcpyHostToDevice, s));
            CUDA_TRY(cudaEventRecord(m->stage_ev[slot], s));
        }
        if (m->opt_timing) CUDA_TRY(cudaEventRecord(m->ev0, s));
        int launches = 0;
        if (n == 1) {
            if (!m->decode_ready) {
                m->build_plan(m->decode, 1, m->opt_fusion != 0);
                m->decode_ready = true;
                m->decode_runs = 0;
            }
            Plan &P = m->decode;
            m->prof_pos = pos;
            if (P.exec && m->opt_graph && !m->opt_profile) {
                CUDA_TRY(cudaGraphLaunch(P.exec, s));
            } else {
                m->run_plan(P);
                ++m->decode_runs;
                if (m->opt_graph && !m->opt_profile && !P.capture_failed) {
                    // capture the step once it has run eagerly (attributes set, no first-use work)
                    P.drop_graph();
                    CUDA_TRY(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
                    for (auto &nd : P.nodes) nd.run(s);
                    cudaError_t e = cudaStreamEndCapture(s, &P.graph);
                    if (e == cudaSuccess) e = cudaGraphInstantiate(&P.exec, P.graph, 0);
                    if (e != cudaSuccess) {
                        // not capturable here: keep running eagerly
                        cudaGetLastError();
                        P.drop_graph();
                        P.capture_failed = true;
                    }
                }
            }
            launches = P.launches();
            m->last_plan = &P;
        } else {
            // resident tensor-core operand planes of the bulk-matmul weights (option tc_planes),
            // decided at the first bulk forward so that decode-only use never holds them
            if (!m->planes_decided) m->build_planes();
            m->build_plan(m->bulk, n, m->opt_fusion != 0);
            m->prof_pos = pos;
            m->run_plan(m->bulk);
            launches = m->bulk.launches();
            m->last_plan = &m->bulk;
            // the bulk frame reused the pool: the decode plan's buffers are handed out again in
            // the same order by its own build, so it stays valid (rebuilt lazily if not)
        }
        if (m->opt_timing) {
            CUDA_TRY(cudaEventRecord(m->ev1, s));
            CUDA_TRY(cudaEventSynchronize(m->ev1));
            float ms = 0.f;
            CUDA_TRY(cudaEventElapsedTime(&ms, m->ev0, m->ev1));
            (n == 1 ? m->tm.last_step_ms : m->tm.last_prefill_ms) = ms;
        }
        m->dev_pos = pos + n;
        m->dev_n = n;
        m->kv_len = pos + n;
        m->tm.n_forward++;
        m->tm.n_launches = launches;
        m->tm.pool_bytes = (int64_t)m->pool.held();
        float *dlog = m->last_plan->regs.at("logits");
        if (logits) {
            if (flags & SYN_LOGITS_ON_DEVICE)
                CUDA_TRY(cudaMemcpyAsync(logits, dlog, (size_t)m->n_vocab * 4, cudaMemcpyDeviceToDevice, s));
            else
                CUDA_TRY(cudaMemcpyAsync(logits, dlog, (size_t)m->n_vocab * 4, cudaMemcpyDeviceToHost, s));
        }
        const bool host_arg = argmax_out && !(flags & SYN_ARGMAX_ON_DEVICE);
        if (argmax_out && !host_arg)
            CUDA_TRY(cudaMemcpyAsync(argmax_out, &m->d_state->argmax, 4, cudaMemcpyDeviceToDevice, s));
        const bool host_out = (logits && !(flags & SYN_LOGITS_ON_DEVICE)) || host_arg;
        if (host_out) {
            // the error bits and the argmax come back with the logits, before one synchronisation
            CUDA_TRY(cudaMemcpyAsync(m->h_out, &m->d_state->err, 4, cudaMemcpyDeviceToHost, s));
            CUDA_TRY(cudaMemcpyAsync(m->h_out + 1, &m->d_state->argmax, 4, cudaMemcpyDeviceToHost, s));
            CUDA_TRY(cudaStreamSynchronize(s));
            if (host_arg) *argmax_out = m->h_out[1];
            const int err = m->h_out[0];
            if (err) {
                CUDA_TRY(cudaMemset(&m->d_state->err, 0, 4));
                if (err & ERR_TC)
                    throw Error{SYN_E_CUDA, "a tensor-core matmul wait timed out (results of this forward are invalid)"};
                if (err & ERR_ATTN)
                    throw Error{SYN_E_CUDA, "an attention copy wait timed out (results of this forward are invalid)"};

                throw Error{SYN_E_INVALID_ARG, "device reported a token id outside the vocabulary"};
            }
        }
    });
}

syn_status syn_logits_device(syn_model *m, const float **ptr, int *n_vocab) {
    return guarded(m, [&] {
        if (!m->finalized || !m->last_plan) throw Error{SYN_E_STATE, "no forward has run"};
        if (ptr) *ptr = m->last_plan->regs.at("logits");
        if (n_vocab) *n_vocab = m->n_vocab;
    });
}

syn_status syn_get_timings(syn_model *m, syn_timings *out) {
    return guarded(m, [&] {
        if (!out) throw Error{SYN_E_INVALID_ARG, "null out"};
        m->tm.pool_bytes = (int64_t)m->pool.held();
        *out = m->tm;
    });
}

syn_status syn_set_option(syn_model *m, const char *key, int64_t value) {
    return guarded(m, [&] {
        if (!key) throw Error{SYN_E_INVALID_ARG, "null key"};
        std::string k = key;
        if (m->stream) CUDA_TRY(cudaStreamSynchronize(m->stream));  // plans may be rebuilt below
        if (k == "fusion") {
            m->opt_fusion = value != 0;
            if (m->finalized) {
                m->build_plan(m->decode, 1, m->opt_fusion != 0);
                m->decode_runs = 0;
                m->invalidate_handle_plans();
            }
        } else if (k == "graph") {
            m->opt_graph = value != 0;
        } else if (k == "timing") {
            m->opt_timing = value != 0;
        } else if (k == "profile") {
            m->opt_profile = value != 0;
        } else if (k == "tc") {
            m->opt_tc = value != 0;
        } else if (k == "tc_planes") {
            if (value < -1 || value > 1) throw Error{SYN_E_INVALID_ARG, "tc_planes must be -1, 0 or 1"};
            m->opt_tc_planes = (int)value;
            m->drop_planes();
            m->planes_decided = false;
            if (m->finalized && value == 1) m->build_planes();
        } else if (k == "attn_tc") {
            m->opt_attn_tc = value != 0;
        } else if (k == "kv_f16") {
            if (m->finalized) throw Error{SYN_E_STATE, "kv_f16 must be set before syn_finalize (it sizes the cache)"};
            m->opt_kv_f16 = value != 0;
        } else if (k == "splits") {
            if (value < 0 || value > 64) throw Error{SYN_E_INVALID_ARG, "splits must be in [0, 64]"};
            m->opt_splits = (int)value;
            if (m->finalized) {
                m->build_plan(m->decode, 1, m->opt_fusion != 0);
                m->decode_runs = 0;
                m->invalidate_handle_plans();
            }
        } else {
            throw Error{SYN_E_INVALID_ARG, "unknown option " + k};
        }
    });
}

syn_status syn_get_info(syn_model *m, const char *key, int64_t *value) {
    return guarded(m, [&] {
        if (!key || !value) throw Error{SYN_E_INVALID_ARG, "null argument"};
        std::string k = key;
        if (k == "n_vocab") *value = m->n_vocab;
        else if (k == "n_embd") *value = m->n_embd;
        else if (k == "n_layer") *value = m->n_layer;
        else if (k == "n_head") *value = m->n_head;
        else if (k == "n_head_kv") *value = m->n_head_kv;
        else if (k == "head_dim") *value = m->head_dim;
        else if (k == "max_ctx") *value = m->max_ctx;
        else if (k == "kv_len") *value = m->kv_len;
        else if (k == "steps_per_layer") *value = (int64_t)m->ad.sec[1].size();
        else if (k == "n_plan_nodes") *value = m->decode_ready ? m->decode.launches() : 0;
        else if (k == "tc_plane_bytes") *value = (int64_t)m->plane_bytes;
        else if (k == "fused") *value = m->any_fused ? 1 : 0;
        else if (k == "kv_f16") *value = m->opt_kv_f16;
        else throw Error{SYN_E_INVALID_ARG, "unknown info key " + k};
    });
}

syn_status syn_debug_write_kv(syn_model *m, int layer, int pos0, int n, const float *k, const float *v) {
    return guarded(m, [&] {
        if (!m->finalized) throw Error{SYN_E_STATE, "before syn_finalize"};
        if (!k || !v || layer < 0 || layer >= m->n_layer || pos0 < 0 || n < 0 || (int64_t)pos0 + n > m->max_ctx || pos0 > m->kv_len)
            throw Error{SYN_E_INVALID_ARG, "bad KV range"};
        const size_t hd = m->head_dim, cnt = (size_t)n * hd;
        std::vector<uint16_t> hk, hv;   // f16 cache: round to nearest on the host
        for (int g = 0; g < m->n_head_kv; ++g) {
            const size_t off = (((size_t)layer * m->n_head_kv + g) * m->max_ctx + pos0) * hd * m->kv_es;
            const float *ks = k + (size_t)g * cnt, *vs = v + (size_t)g * cnt;
            const void *ksrc = ks, *vsrc = vs;
            if (m->kv_es == 2) {
                hk.resize(cnt);
                hv.resize(cnt);
                for (size_t i = 0; i < cnt; ++i) {
                    hk[i] = f32_bits_to_half_bits(ks[i]);
                    hv[i] = f32_bits_to_half_bits(vs[i]);
                }
                ksrc = hk.data();
                vsrc = hv.data();
            }
            CUDA_TRY(cudaMemcpy(static_cast<uint8_t *>(m->kcache) + off, ksrc, cnt * m->kv_es, cudaMemcpyHostToDevice));
            CUDA_TRY(cudaMemcpy(static_cast<uint8_t *>(m->vcache) + off, vsrc, cnt * m->kv_es, cudaMemcpyHostToDevice));
        }
        CUDA_TRY(cudaStreamSynchronize(m->stream));
        m->kv_len = std::max(m->kv_len, pos0 + n);
    });
}

syn_status syn_debug_read_kv(syn_model *m, int layer, int pos0, int n, float *k, float *v) {
    return guarded(m, [&] {
        if (!m->finalized) throw Error{SYN_E_STATE, "before syn_finalize"};
        if (!k || !v || layer < 0 || layer >= m->n_layer || pos0 < 0 || n < 0 || (int64_t)pos0 + n > m->max_ctx)
            throw Error{SYN_E_INVALID_ARG, "bad KV range"};
        CUDA_TRY(cudaStreamSynchronize(m->stream));
        const size_t hd = m->head_dim, cnt = (size_t)n * hd;
        std::vector<uint16_t> hk(m->kv_es == 2 ? cnt : 0), hv(m->kv_es == 2 ? cnt : 0);
        for (int g = 0; g < m->n_head_kv; ++g) {
            const size_t off = (((size_t)layer * m->n_head_kv + g) * m->max_ctx + pos0) * hd * m->kv_es;
            float *kd = k + (size_t)g * cnt, *vd = v + (size_t)g * cnt;
            if (m->kv_es == 2) {
                CUDA_TRY(cudaMemcpy(hk.data(), static_cast<const uint8_t *>(m->kcache) + off, cnt * 2, cudaMemcpyDeviceToHost));
                CUDA_TRY(cudaMemcpy(hv.data(), static_cast<const uint8_t *>(m->vcache) + off, cnt * 2, cudaMemcpyDeviceToHost));
                for (size_t i = 0; i < cnt; ++i) {
                    kd[i] = __half2float(__ushort_as_half(hk[i]));
                    vd[i] = __half2float(__ushort_as_half(hv[i]));
                }
            } else {
                CUDA_TRY(cudaMemcpy(kd, static_cast<const uint8_t *>(m->kcache) + off, cnt * 4, cudaMemcpyDeviceToHost));
                CUDA_TRY(cudaMemcpy(vd, static_cast<const uint8_t *>(m->vcache) + off, cnt * 4, cudaMemcpyDeviceToHost));
            }
        }
    });
}

syn_status syn_debug_read_register(syn_model *m, const char *name, float *out, int count) {
    return guarded(m, [&] {
        if (!m->last_plan) throw Error{SYN_E_STATE, "no forward has run"};
        if (!name || !out) throw Error{SYN_E_INVALID_ARG, "null argument"};
        const std::string r = name;
        if (m->last_plan->folded.count(r))
            throw Error{SYN_E_STATE, "register " + r + " was folded away by the fusion pass"};
        auto it = m->last_plan->regs.find(r);
        if (it == m->last_plan->regs.end()) throw Error{SYN_E_INVALID_ARG, "no register " + r};
        if (count < 0 || count > m->reg_width.at(r)) throw Error{SYN_E_INVALID_ARG, "count exceeds register width"};
        CUDA_TRY(cudaStreamSynchronize(m->stream));
        CUDA_TRY(cudaMemcpy(out, it->second, (size_t)count * 4, cudaMemcpyDeviceToHost));
    });
}

syn_status syn_debug_dequant(syn_model *m, const char *gguf_name, int row0, int nrows, float *out) {
    return guarded(m, [&] {
        if (!gguf_name || !out) throw Error{SYN_E_INVALID_ARG, "null argument"};
        auto it = m->tensors.find(gguf_name);
        if (it == m->tensors.end()) throw Error{SYN_E_MISSING_TENSOR, std::string("no tensor ") + gguf_name};
        const DevMatrix &W = it->second.mat;
        if (row0 < 0 || nrows < 0 || row0 + nrows > W.N) throw Error{SYN_E_INVALID_ARG, "row range"};
        float *d = nullptr;
        const size_t bytes = (size_t)nrows * W.K * 4;
        CUDA_TRY(cudaMalloc(&d, std::max<size_t>(bytes, 4)));
        launch_dequant_rows(W, row0, nrows, d, m->stream);
        cudaError_t e = cudaStreamSynchronize(m->stream);
        if (e == cudaSuccess) e = cudaMemcpy(out, d, bytes, cudaMemcpyDeviceToHost);
        cudaFree(d);
        if (e != cudaSuccess) throw Error{SYN_E_CUDA, cudaGetErrorString(e)};
    });
}

syn_status syn_get_profile(syn_model *m, char *buf, size_t len, int reset) {
    return guarded(m, [&] {
        if (!buf || !len) throw Error{SYN_E_INVALID_ARG, "null buffer"};
        std::string out;
        char line[256];
        for (auto &e : m->prof) {
            std::snprintf(line, sizeof line, "%s %lld %.6f %.0f %.0f\n", e.first.c_str(), (long long)e.second.launches,
                          e.second.ms, e.second.bytes, e.second.flops);
            out += line;
        }
        if (out.size() + 1 > len) throw Error{SYN_E_INVALID_ARG, "buffer too small: need " + std::to_string(out.size() + 1)};
        std::memcpy(buf, out.c_str(), out.size() + 1);
        if (reset) m->prof.clear();
    });
}

const char *syn_last_error(const syn_model *m) { return m ? m->err.c_str() : "null model"; }

syn_status syn_kv_create(syn_model *m, syn_kv **out) {
    if (!out) return SYN_E_INVALID_ARG;
    *out = nullptr;
    return guarded(m, [&] {
        if (!m->finalized) throw Error{SYN_E_STATE, "syn_kv_create before syn_finalize"};
        syn_kv *h = new (std::nothrow) syn_kv();
        if (!h) throw Error{SYN_E_OOM, "KV handle"};
        h->m = m;
        const size_t kv = (size_t)m->n_layer * m->n_head_kv * m->max_ctx * m->head_dim * m->kv_es;
        cudaError_t e = cudaMalloc(&h->kcache, kv);
        if (e == cudaSuccess) e = cudaMalloc(&h->vcache, kv);
        if (e == cudaSuccess) e = cudaMalloc(&h->d_state, sizeof(DevState));
        if (e == cudaSuccess) e = cudaMemset(h->kcache, 0, kv);
        if (e == cudaSuccess) e = cudaMemset(h->vcache, 0, kv);
        if (e == cudaSuccess) e = cudaMemset(h->d_state, 0, sizeof(DevState));
        if (e != cudaSuccess) {
            h->release();
            delete h;
            throw Error{SYN_E_OOM, "KV handle: cudaMalloc of 2 x " + std::to_string(kv) + " bytes failed"};
        }
        m->handles.insert(h);
        *out = h;
    });
}

syn_status syn_kv_select(syn_model *m, syn_kv *kv) {
    return guarded(m, [&] {
        if (kv && (kv->m != m || !m->handles.count(kv))) throw Error{SYN_E_INVALID_ARG, "KV handle of another model"};
        if (m->active == kv) return;
        if (m->active) m->swap_kv(m->active);   // the selected handle takes its state back
        if (kv) m->swap_kv(kv);                 // and the new one lends its state to the model
        m->active = kv;
        m->last_plan = nullptr;
    });
}

void syn_kv_destroy(syn_kv *kv) {
    if (!kv) return;
    syn_model *m = kv->m;
    if (m) {
        if (m->stream) cudaStreamSynchronize(m->stream);
        if (m->active == kv) syn_kv_select(m, nullptr);
        m->handles.erase(kv);
        kv->release();
    }
    delete kv;
}

void syn_destroy(syn_model *m) {
    if (!m) return;
    if (m->stream) cudaStreamSynchronize(m->stream);
    delete m;
}

}  // extern "C"
