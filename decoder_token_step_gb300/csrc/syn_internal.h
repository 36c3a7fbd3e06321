// syn_internal.h -- types shared by the host runtime and the CUDA kernels of libsyn.
//
// Nothing here is part of the public ABI (include/syn.h). Kernel launchers are plain C++ functions
// that take a parameter struct and a stream; the runtime calls them while recording a step plan.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include <cuda_runtime.h>

namespace syn {

// ---------------------------------------------------------------------------------------------
// Weight storage on the device.
//
// A GGUF matrix has ne0 = K (in-features, contiguous) and ne1 = N rows. At load time the GGUF
// blocks are split into two arrays so that every row of codes is 16-byte aligned for 128-bit
// loads ("structure of arrays"; the bytes and the dequantised values are unchanged):
//   F32  : codes = float [N][K]
//   F16  : codes = half  [N][K]
//   Q8_0 : codes = uint8 [N][K] offset-binary (q + 128), scales = half [N][K/32]   (w = d * q)
//   Q4_0 : codes = uint8 [N][K/2], scales = half [N][...]  (byte j of a 16-byte block holds
//          element j in its low nibble and element j+16 in its high nibble; w = d * (code - 8))
// Every row of codes is padded with zero bytes to a multiple of 32 bytes (one 256-bit load), and
// the scales of a row are padded with zero scales to match, so padding decodes to exactly 0.
// ---------------------------------------------------------------------------------------------
enum WType : int { W_F32 = 0, W_F16 = 1, W_Q4_0 = 2, W_Q8_0 = 8 };

struct DevMatrix {
    int wtype = W_F32;
    int64_t K = 0;              // in-features (ne0)
    int64_t N = 0;              // rows (ne1); 1 for vectors
    const void *codes = nullptr;
    const uint16_t *scales = nullptr;  // f16 bits, quantised types only
    size_t row_bytes = 0;       // bytes of one row of codes (multiple of 32)
    int64_t scale_stride = 0;   // scales per row (>= K/32)
};

// ---------------------------------------------------------------------------------------------
// Step state kept in device memory so that a captured decode graph can be replayed unchanged:
// the kernels read the position from here, and the last kernel of a step advances it.
// ---------------------------------------------------------------------------------------------
struct DevState {
    int pos;        // absolute position of row 0 of the current forward
    int n;          // rows of the current forward
    int err;        // sticky device-side error bits (see ERR_*)
    int argmax;     // index of the largest logit of the last forward
};
enum : int { ERR_TOKEN_RANGE = 1, ERR_CTX = 2, ERR_TC = 8, ERR_ATTN = 16 };

// ---------------------------------------------------------------------------------------------
// Launch parameter structs
// ---------------------------------------------------------------------------------------------
enum Epi : int { EPI_STORE = 0, EPI_ADD = 1 };  // y = W x  /  y += W x
enum Act : int { ACT_NONE = 0, ACT_SILU = 1, ACT_GELU = 2, ACT_GELU_TANH = 3, ACT_RELU = 4 };

struct GemvSeg {
    DevMatrix W;
    float *out = nullptr;          // N floats per input row (row stride ldo)
    const float *bias = nullptr;   // optional, N floats, added before the epilogue
    int epi = EPI_STORE;
    int64_t ldo = 0;
};

// y = W . prologue(x) for up to 3 matrices sharing the input (fused Q/K/V), or the gated form
// out = act(Wg . h) * (Wu . h) when gate_up is set (seg[0] = gate, seg[1] = up, output seg[0]).
struct GemvParams {
    GemvSeg seg[3];
    int nseg = 1;
    const float *x = nullptr;      // input rows, row stride ldx
    int64_t ldx = 0;
    int rows = 1;                  // input rows (bs or bulk rows); decode uses 1
    const float *norm_w = nullptr; // prologue rms_norm weight (K floats) or nullptr
    float eps = 0.f;
    int gate_up = 0;
    int act = ACT_NONE;
    int gend[3] = {0, 0, 0};       // GEMV row groups before the end of segment i, cumulative (set by the launcher)
};

// Optional post-branch update in a decode GEMV's prologue, before its norm: x_new = x + t / rms(t) * w,
// written to out (each CTA its slice; out != the GEMV's x), and the matmul reads x_new. A separate
// kernel argument, so that the GEMV without it keeps its parameter block.
struct GemvPre {
    const float *t = nullptr;
    const float *w = nullptr;
    float *out = nullptr;
};

// fill p.gend: cumulative counts of kr-row groups per segment; unused segments repeat the total, so
// that a group index below the total never selects them
inline void gemv_set_groups(GemvParams &p, int kr) {
    int acc = 0;
    for (int i = 0; i < 3; ++i) {
        if (i < p.nseg && !p.gate_up) acc += (int)((p.seg[i].W.N + kr - 1) / kr);
        p.gend[i] = acc;
    }
}

struct EmbedParams {
    DevMatrix E;
    const int *tokens = nullptr;
    int n = 1;
    float *out = nullptr;          // [n][K]
    float scale = 1.f;             // folded `scale` step (1 = none)
    DevState *state = nullptr;
};

struct RmsParams {
    const float *x = nullptr; float *y = nullptr; const float *w = nullptr;
    int rows = 1, width = 0; int64_t ld = 0; float eps = 0.f;
    float *residual = nullptr;     // when set: residual += rms_norm(x) * w  (y unused)
};

enum EltOp : int { ELT_ACT = 0, ELT_MUL = 1, ELT_ADD = 2, ELT_SCALE = 3, ELT_COPY = 4, ELT_BIAS = 5, ELT_ACT_MUL = 6 };  // ACT_MUL: act(a) * b
struct EltParams {
    float *y = nullptr; const float *a = nullptr; const float *b = nullptr;
    int rows = 1, width = 0; int64_t ld = 0; int op = ELT_COPY; int act = ACT_NONE; float c = 1.f;
};

// Per-head transforms of q and k before attention, and the K/V append, in the archdef's order:
// [add_bias] -> [norm_heads] -> rope. Either half can be disabled (unfused path uses one op at a
// time through the same kernel).
struct HeadsParams {
    float *q = nullptr; int nq = 0;            // q heads (0: none)
    float *k = nullptr; int nk = 0;            // k heads (0: none)
    const float *v = nullptr;                  // v rows to append (with kcache)
    int64_t ldq = 0, ldk = 0, ldv = 0;
    int hd = 0, rows = 1;
    const float *bq = nullptr, *bk = nullptr, *bv = nullptr;   // biases
    const float *wq = nullptr, *wk = nullptr;                  // norm_heads weights (hd floats)
    int rope_q = 0, rope_k = 0, rope_adjacent = 0;
    const float2 *rope_cs = nullptr;           // [max_ctx][hd/2] (cos, sin)
    float eps = 0.f;
    void *kcache = nullptr, *vcache = nullptr; // layer base [n_kv][max_ctx][hd] (f32, or f16 when kv_f16); nullptr: no append
    int max_ctx = 0;
    int kv_f16 = 0;                            // the cache stores f16 (rounded to nearest)
    const DevState *state = nullptr;
};

struct AttnParams {
    const float *q = nullptr; int64_t ldq = 0;   // [rows][n_head*hd]
    float *out = nullptr; int64_t ldo = 0;       // [rows][n_head*hd]
    const void *kcache = nullptr, *vcache = nullptr;   // layer base [n_kv][max_ctx][hd], f32 (or f16: kv_f16)
    int kv_f16 = 0;
    int n_head = 0, n_kv = 0, hd = 0, max_ctx = 0, rows = 1;
    int window = 0;                 // 0 = global; else keys t > p - window
    int splits = 1;                 // split-K count (grid.y)
    float *part = nullptr;          // scratch: [rows][n_head][splits][hd + 4] (o, m, l, pad)
    unsigned *counters = nullptr;   // [rows][n_kv] completion counters, zero between launches
    const DevState *state = nullptr;
    int *err = nullptr;             // where a timed-out wait records ERR_ATTN (DevState::err)
    int spin = -1;                  // polls before a wait gives up (-1: the default bound; 0: at once)
    // decode (rows == 1) with the per-head transforms folded in: q is read untransformed and each
    // CTA transforms its group's heads in registers; the CTA whose key slice holds the new position
    // transforms that position's k, adds the v bias and appends both to the cache (heads.q/k/v are
    // the raw projections; heads.kcache/vcache/max_ctx as in kcache/vcache)
    int fuse_heads = 0;
    HeadsParams heads;
};

struct ArgmaxParams {
    const float *x = nullptr; int n = 0;
    float *part_v = nullptr; int *part_i = nullptr; unsigned *counter = nullptr;
    DevState *state = nullptr; int advance = 0;   // advance state->pos by state->n when done
};

struct GemmParams {          // bulk rows: Y[r][j] (+)= sum_k W[j][k] X[r][k]
    GemvParams g;            // reuses the segment/prologue description; g.rows = M
};

// Sets a kernel's dynamic shared-memory limit (cudaFuncAttributeMaxDynamicSharedMemorySize) on the
// calling thread's current device, once per (kernel, device, size): the attribute is per device.
// Thread-safe; never called during a stream capture (the first launch of every kernel of a plan
// runs eagerly).
cudaError_t ensure_dyn_smem(const void *func, int bytes);

// launchers (stream-ordered, no synchronisation)
void launch_gemv(const GemvParams &p, int sm_count, cudaStream_t s, const GemvPre *pre = nullptr);
void launch_gemm_rows(const GemvParams &p, cudaStream_t s);
// bulk rows on the tensor cores (k_gemm_tc.cu): supported shapes, scratch sizes, launch (returns the
// launch error; a timed-out wait inside sets ERR_TC in *err)
bool gemm_tc_supported(const GemvParams &p);
size_t gemm_tc_x_bytes(const GemvParams &p);
size_t gemm_tc_w_bytes(const GemvParams &p);
// the resident operand planes of one weight matrix (bytes; and the conversion into `planes`)
size_t gemm_tc_planes_bytes(const DevMatrix &W);
cudaError_t launch_dequant_split(const DevMatrix &W, void *planes, cudaStream_t s);
// planes[i]: resident operand planes of segment i's weight ([Wh N*K f16][Wl N*K f16][1/scale per row
// N f32], converted once), or nullptr to convert into wscratch now.
cudaError_t launch_gemm_tc(const GemvParams &p, const void *const planes[3], void *xscratch, void *wscratch, int *err,
                           cudaStream_t s);
void launch_embed(const EmbedParams &p, cudaStream_t s);
void launch_rmsnorm(const RmsParams &p, cudaStream_t s);
void launch_eltwise(const EltParams &p, cudaStream_t s);
void launch_heads(const HeadsParams &p, cudaStream_t s);
void launch_attention(const AttnParams &p, cudaStream_t s);
// same kernel without programmatic dependent launch: it starts only after the previous work on the
// stream has completed (for callers whose preceding kernel writes the state it reads first)
void launch_attention_ordered(const AttnParams &p, cudaStream_t s);
// bulk-prefill attention on the tensor cores (k_attn_tc.cu): supported shapes (rows > 1, head size
// 64 or 128), scratch sizes (the q planes depend on rows, the K/V planes on max_ctx), launch of the
// split kernels and the attention (returns the launch error; a timed-out wait sets ERR_ATTN in *p.err)
bool attention_tc_supported(const AttnParams &p);
size_t attention_tc_q_bytes(const AttnParams &p);
size_t attention_tc_kv_bytes(const AttnParams &p);
cudaError_t launch_attention_tc(const AttnParams &p, void *qscratch, void *kvscratch, cudaStream_t s);
void launch_argmax(const ArgmaxParams &p, int blocks, cudaStream_t s);
void launch_copy_row(float *dst, const float *src, int width, cudaStream_t s);
void launch_dequant_rows(const DevMatrix &W, int row0, int nrows, float *out, cudaStream_t s);

// ---------------------------------------------------------------------------------------------
// .archdef text (host)
// ---------------------------------------------------------------------------------------------
struct Step {
    int line = 0;
    std::string dst;               // register assigned (or modified, in the in-place form)
    std::string op;
    std::vector<std::string> args; // in the in-place form args[0] == dst
    bool assign = false;           // "dst = op(...)" form
};

struct Archdef {
    std::string arch;
    int window_pattern = 0;
    int rope_adjacent = 0;
    std::vector<Step> sec[3];      // prologue, block, epilogue
};

// SHA-256 of a byte string as 64 lower-case hex digits (sha256.cpp).
std::string sha256_hex(const void *data, size_t len);

// Parse and validate; on failure returns false and fills err with "file: line N: message".
bool parse_archdef(const std::string &file_arch, const std::string &text, Archdef &out, std::string &err);
extern const char *const kOps[16];

}  // namespace syn
