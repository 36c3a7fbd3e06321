/*
 * oracle.c -- the CPU oracle of the decoder token step.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT. Only the tests, the smoke check and the bench's
 * CPU-baseline leg may build, load or call this file. It shares no code, header, table or helper
 * with the CUDA library; the only thing both sides see is the seeded input bytes.
 *
 * What it computes: the per-token forward of a GGUF decoder exactly as an .archdef text spells it
 * out ("Local inference and architectures", synsema.dev, sections "The format" and "The
 * operations"): a prologue, a block run once per layer with {i} replaced by the layer index, and
 * an epilogue, over named registers. Token-by-token prefill, decode and bulk prefill all go through
 * the same function ("Execution contract", cyber.page, section "Forward phase / Text generation");
 * the KV cache is sized to the maximum context, appended to on every call and cleared by
 * orc_reset_kv ("Execution contract", section "Memory lifecycle / KV cache").
 *
 * Precision. The pages' engine multiplies in f32 ("Local inference and architectures", section
 * "Choosing the engine"). Here every register and the KV cache hold f32 values; each op forms its
 * result in double (a product of two floats is exact in double) and rounds it to f32 once when it
 * stores it. Reductions (dot products, sums of squares, softmax sums) therefore carry no
 * order-dependent f32 rounding, and the CUDA path's summation order is free.
 *
 * Speed is not a goal: loops run in index order, weights are dequantised row by row on the fly
 * straight from the GGUF block bytes, and the only parallelism is OpenMP over independent output
 * rows of a matmul, which does not change any result.
 */
#include <ctype.h>
#include <math.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR 1

#define MAX_STEPS 96
#define MAX_ARGS 6
#define MAX_REGS 32
#define MAX_META 96
#define NAME_LEN 160

/* GGUF tensor type ids */
enum { T_F32 = 0, T_F16 = 1, T_Q4_0 = 2, T_Q8_0 = 8 };

/* ------------------------------------------------------------------------------------------ */
/* f32 -> nearest binary16 value (returned as f32), ties to even: the representable halves are   */
/* the multiples of 2^(e-10) in [2^e, 2^(e+1)) for e >= -14 and the multiples of 2^-24 below   */
/* 2^-14; the largest finite half is 65504, and anything that rounds above it is infinite. Used */
/* only when the cache is configured to store f16 keys and values.                               */
/* ------------------------------------------------------------------------------------------ */
static float round_to_half(float f) {
    if (isnan(f) || isinf(f)) return f;
    double a = fabs((double)f);
    if (a == 0.0) return f;
    int e2;
    frexp(a, &e2);                 /* a in [2^(e2-1), 2^e2) */
    int lead = e2 - 1;             /* exponent of the leading bit */
    double quantum = lead < -14 ? ldexp(1.0, -24) : ldexp(1.0, lead - 10);
    double r = nearbyint(a / quantum) * quantum;   /* default rounding mode: to nearest, ties even */
    if (r > 65504.0) r = INFINITY;
    return (float)(f < 0 ? -r : r);
}

/* ------------------------------------------------------------------------------------------ */
/* f16 -> f32, written from the IEEE 754 binary16 definition: sign, 5-bit exponent (bias 15),   */
/* 10-bit fraction; exponent 0 is subnormal (fraction * 2^-24), 31 is inf/NaN.                  */
/* ------------------------------------------------------------------------------------------ */
static float half_to_float(uint16_t h) {
    int sign = (h >> 15) & 1;
    int exp = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (exp == 0)
        v = ldexp((double)frac, -24);
    else if (exp == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(frac | 0x400), exp - 25);
    return (float)(sign ? -v : v);
}

/*
 * Dequantise elements [0, k) of one row of a GGUF tensor into out (f32).
 * Block layouts (GGUF storage formats, not given by the pages):
 *   f32  : 4-byte IEEE floats.
 *   f16  : 2-byte IEEE halves.
 *   Q8_0 : 34-byte blocks of 32 weights {f16 d; int8 q[32]}, w[j] = d * q[j].
 *   Q4_0 : 18-byte blocks of 32 weights {f16 d; uint8 qs[16]}, w[j] = d * ((qs[j] & 15) - 8) and
 *          w[j + 16] = d * ((qs[j] >> 4) - 8) for j < 16.
 * The product d * code is formed in f32 (it is exact: at most 11 + 8 significant bits).
 */
static void dequant_row(int type, const uint8_t *row, int64_t k, float *out) {
    if (type == T_F32) {
        memcpy(out, row, (size_t)k * 4);
    } else if (type == T_F16) {
        for (int64_t j = 0; j < k; ++j) {
            uint16_t h;
            memcpy(&h, row + 2 * j, 2);
            out[j] = half_to_float(h);
        }
    } else if (type == T_Q8_0) {
        for (int64_t b = 0; b < k / 32; ++b) {
            const uint8_t *blk = row + 34 * b;
            uint16_t hd;
            memcpy(&hd, blk, 2);
            float d = half_to_float(hd);
            for (int j = 0; j < 32; ++j) out[32 * b + j] = d * (float)(int8_t)blk[2 + j];
        }
    } else if (type == T_Q4_0) {
        for (int64_t b = 0; b < k / 32; ++b) {
            const uint8_t *blk = row + 18 * b;
            uint16_t hd;
            memcpy(&hd, blk, 2);
            float d = half_to_float(hd);
            for (int j = 0; j < 16; ++j) {
                out[32 * b + j] = d * (float)((blk[2 + j] & 15) - 8);
                out[32 * b + j + 16] = d * (float)((blk[2 + j] >> 4) - 8);
            }
        }
    }
}

static size_t row_bytes(int type, int64_t k) {
    switch (type) {
    case T_F32: return (size_t)k * 4;
    case T_F16: return (size_t)k * 2;
    case T_Q8_0: return (size_t)(k / 32) * 34;
    case T_Q4_0: return (size_t)(k / 32) * 18;
    }
    return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* Elementwise ops ("Local inference and architectures", section "The operations").            */
/* ------------------------------------------------------------------------------------------ */
static double op_silu(double x) { return x / (1.0 + exp(-x)); }
/* exact GELU: x * Phi(x), Phi the standard normal CDF */
static double op_gelu(double x) { return 0.5 * x * (1.0 + erf(x / sqrt(2.0))); }
/* tanh approximation of GELU (PyTorch's approximate="tanh") */
static double op_gelu_tanh(double x) {
    const double c = sqrt(2.0 / M_PI);
    return 0.5 * x * (1.0 + tanh(c * (x + 0.044715 * x * x * x)));
}
static double op_relu(double x) { return x > 0.0 ? x : 0.0; }

/* y = x / sqrt(mean(x^2) + eps) * w over n elements: the rms_norm operation ("Local inference and
 * architectures", section "The operations"), w the stored norm weight, eps read from the GGUF
 * metadata key <arch>.attention.layer_norm_rms_epsilon. */
static void rms_norm_vec(const float *x, const float *w, int n, double eps, float *y) {
    double ss = 0.0;
    for (int j = 0; j < n; ++j) ss += (double)x[j] * (double)x[j];
    double inv = 1.0 / sqrt(ss / n + eps);
    for (int j = 0; j < n; ++j) y[j] = (float)((double)x[j] * inv * (double)w[j]);
}

/*
 * Rotary position embedding of one head of length hd at absolute position p: the rope operation
 * ("Local inference and architectures", section "The operations"; the cos/sin of p * theta_j are
 * what "Execution contract", section "Position caches", precomputes per position).
 * Frequencies theta_j = base^(-2j/hd), j < hd/2, base from <arch>.rope.freq_base; the angle is
 * p * theta_j. pairs_adjacent: rotate (2j, 2j+1); otherwise rotate (j, j + hd/2). The pairing is
 * not GGUF metadata: the definition states it (`param rope_pairs adjacent`, llama).
 */
static void rope_head(float *v, int hd, int64_t p, double base, int pairs_adjacent) {
    for (int j = 0; j < hd / 2; ++j) {
        double theta = pow(base, -2.0 * j / hd);
        double ang = (double)p * theta;
        double c = cos(ang), s = sin(ang);
        int i0 = pairs_adjacent ? 2 * j : j;
        int i1 = pairs_adjacent ? 2 * j + 1 : j + hd / 2;
        double a = v[i0], b = v[i1];
        v[i0] = (float)(a * c - b * s);
        v[i1] = (float)(a * s + b * c);
    }
}

/*
 * Attention of one query head q[hd] over keys/values t in [t0, t1] (inclusive), cache rows of
 * stride hd: o = sum_t softmax_t(q.K_t / sqrt(hd)) V_t, softmax with the max subtracted. The
 * attention operation ("Local inference and architectures", section "The operations") over the
 * cache that every step appends to ("Execution contract", section "Memory lifecycle / KV cache");
 * the caller picks [t0, t1]: t1 = the query's position, t0 = 0, or t1 - window + 1 on the
 * sliding-window layers (section "Rules").
 */
static void attend_head(const float *q, const float *K, const float *V, int hd, int64_t t0,
                        int64_t t1, float *o) {
    int64_t n = t1 - t0 + 1;
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    double scale = 1.0 / sqrt((double)hd), mx = -INFINITY;
    for (int64_t t = t0; t <= t1; ++t) {
        double d = 0.0;
        for (int j = 0; j < hd; ++j) d += (double)q[j] * (double)K[t * hd + j];
        s[t - t0] = d * scale;
        if (s[t - t0] > mx) mx = s[t - t0];
    }
    double sum = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        s[t] = exp(s[t] - mx);
        sum += s[t];
    }
    for (int j = 0; j < hd; ++j) {
        double acc = 0.0;
        for (int64_t t = t0; t <= t1; ++t) acc += s[t - t0] * (double)V[t * hd + j];
        o[j] = (float)(acc / sum);
    }
    free(s);
}

/* ------------------------------------------------------------------------------------------ */
/* Model state                                                                                 */
/* ------------------------------------------------------------------------------------------ */
typedef struct {
    int line;
    char dst[32]; /* register assigned or modified */
    char op[24];
    int nargs;
    char args[MAX_ARGS][NAME_LEN]; /* in the in-place form args[0] == dst */
} step_t;

typedef struct {
    char name[NAME_LEN];
    int type;
    int64_t ne[4];
    int ndims;
    const uint8_t *data; /* borrowed: the caller keeps the bytes alive */
} tensor_t;

typedef struct {
    char name[32];
    int rows, width;
    float *v; /* rows * width */
} reg_t;

typedef struct orc_model {
    char arch[32];
    char meta_k[MAX_META][96];
    char meta_v[MAX_META][64];
    int n_meta;
    int window_pattern;
    int rope_adjacent;
    step_t steps[3][MAX_STEPS]; /* prologue, block, epilogue */
    int n_steps[3];
    tensor_t *tensors;
    int n_tensors, cap_tensors;
    reg_t regs[MAX_REGS];
    int n_regs;
    /* hyper-parameters read from metadata */
    int n_layer, n_embd, n_head, n_head_kv, head_dim, window;
    double eps, rope_base;
    int64_t max_ctx, kv_len;
    float **K, **V; /* per layer [n_head_kv][max_ctx][head_dim] */
    int kv_f16;     /* the cache stores keys and values rounded to f16 (a configuration, off by default) */
    char err[512];
} orc_model;

static int fail(orc_model *m, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(m->err, sizeof m->err, fmt, ap);
    va_end(ap);
    return ORC_ERR;
}

static const char *meta_get(orc_model *m, const char *key) {
    for (int i = 0; i < m->n_meta; ++i)
        if (!strcmp(m->meta_k[i], key)) return m->meta_v[i];
    return NULL;
}

/* Look a name up as "<arch>.<name>", "<arch>.attention.<name>", "<arch>.rope.<name>". */
static const char *meta_arch(orc_model *m, const char *name) {
    static const char *pre[] = {"", "attention.", "rope."};
    char key[160];
    for (int i = 0; i < 3; ++i) {
        snprintf(key, sizeof key, "%s.%s%s", m->arch, pre[i], name);
        const char *v = meta_get(m, key);
        if (v) return v;
    }
    return NULL;
}

static char *trim(char *s) {
    while (isspace((unsigned char)*s)) ++s;
    char *e = s + strlen(s);
    while (e > s && isspace((unsigned char)e[-1])) *--e = 0;
    return s;
}

static const char *OPS[] = {"embed", "rms_norm", "matmul", "add_bias", "norm_heads", "rope",
                            "attention", "silu", "gelu", "gelu_tanh", "relu", "mul",
                            "add", "scale", "copy", "last"};

static int is_op(const char *s) {
    for (size_t i = 0; i < sizeof OPS / sizeof OPS[0]; ++i)
        if (!strcmp(OPS[i], s)) return 1;
    return 0;
}

/*
 * Parse an .archdef text ("Local inference and architectures", sections "The format" and
 * "Rules"): "arch NAME", "kind decoder", optional "param KEY VALUE" lines, then the sections
 * prologue / block / epilogue, each a list of "dst = op(args)" or "op(dst, args)" lines;
 * '#' starts a comment, blank lines are ignored.
 */
static int parse_archdef(orc_model *m, const char *file_arch, const char *text) {
    int section = -1, line_no = 0, have_arch = 0;
    char buf[1024];
    for (const char *p = text; *p;) {
        const char *nl = strchr(p, '\n');
        size_t len = nl ? (size_t)(nl - p) : strlen(p);
        ++line_no;
        if (len >= sizeof buf) return fail(m, "line %d: line too long", line_no);
        memcpy(buf, p, len);
        buf[len] = 0;
        p = nl ? nl + 1 : p + len;
        char *line = buf;
        char *hash = strchr(line, '#');
        if (hash) *hash = 0;
        char *s = trim(line);
        if (!*s) continue;
        if (!strncmp(s, "arch ", 5)) {
            snprintf(m->arch, sizeof m->arch, "%s", trim(s + 5));
            have_arch = 1;
            continue;
        }
        if (!strncmp(s, "kind ", 5)) {
            if (strcmp(trim(s + 5), "decoder")) { return fail(m, "line %d: kind must be decoder", line_no); }
            continue;
        }
        if (!strncmp(s, "param ", 6)) {
            char key[64], val[64];
            if (sscanf(s + 6, "%63s %63s", key, val) != 2) { return fail(m, "line %d: bad param", line_no); }
            if (!strcmp(key, "window_pattern")) m->window_pattern = atoi(val);
            else if (!strcmp(key, "rope_pairs")) m->rope_adjacent = !strcmp(val, "adjacent");
            else { return fail(m, "line %d: unknown param %s", line_no, key); }
            continue;
        }
        if (!strcmp(s, "prologue")) { section = 0; continue; }
        if (!strcmp(s, "block")) { section = 1; continue; }
        if (!strcmp(s, "epilogue")) { section = 2; continue; }
        if (section < 0) { return fail(m, "line %d: statement outside a section", line_no); }
        step_t st;
        memset(&st, 0, sizeof st);
        st.line = line_no;
        char *eq = strchr(s, '=');
        char *call = s;
        if (eq) {
            *eq = 0;
            snprintf(st.dst, sizeof st.dst, "%.31s", trim(s));
            call = trim(eq + 1);
        }
        char *lp = strchr(call, '('), *rp = strrchr(call, ')');
        if (!lp || !rp || rp < lp) { return fail(m, "line %d: expected op(args)", line_no); }
        *lp = 0;
        *rp = 0;
        snprintf(st.op, sizeof st.op, "%s", trim(call));
        if (!is_op(st.op)) { return fail(m, "line %d: unknown operation %s", line_no, st.op); }
        char *argsave = NULL;
        for (char *a = strtok_r(lp + 1, ",", &argsave); a; a = strtok_r(NULL, ",", &argsave)) {
            if (st.nargs == MAX_ARGS) { return fail(m, "line %d: too many arguments", line_no); }
            snprintf(st.args[st.nargs++], NAME_LEN, "%s", trim(a));
        }
        if (!eq) {
            if (st.nargs == 0) { return fail(m, "line %d: in-place op needs a register", line_no); }
            snprintf(st.dst, sizeof st.dst, "%.31s", st.args[0]);
        }
        if (m->n_steps[section] == MAX_STEPS) { return fail(m, "too many steps"); }
        m->steps[section][m->n_steps[section]++] = st;
    }
    if (!have_arch) return fail(m, "no arch line");
    if (file_arch && *file_arch && strcmp(file_arch, m->arch))
        return fail(m, "file %s.archdef declares arch %s", file_arch, m->arch);
    return ORC_OK;
}

static reg_t *reg_find(orc_model *m, const char *name) {
    for (int i = 0; i < m->n_regs; ++i)
        if (!strcmp(m->regs[i].name, name)) return &m->regs[i];
    return NULL;
}

/* (Re)shape a register, keeping no contents. */
static reg_t *reg_set(orc_model *m, const char *name, int rows, int width) {
    reg_t *r = reg_find(m, name);
    if (!r) {
        r = &m->regs[m->n_regs++];
        memset(r, 0, sizeof *r);
        snprintf(r->name, sizeof r->name, "%s", name);
    }
    free(r->v);
    r->rows = rows;
    r->width = width;
    r->v = (float *)calloc((size_t)rows * width, sizeof(float));
    return r;
}

static tensor_t *tensor_find(orc_model *m, const char *name) {
    for (int i = 0; i < m->n_tensors; ++i)
        if (!strcmp(m->tensors[i].name, name)) return &m->tensors[i];
    return NULL;
}

/* Resolve "a | b" (first present tensor, "Local inference and architectures", "Rules") with
 * {i} replaced by the layer index. */
static tensor_t *tensor_arg(orc_model *m, const char *arg, int layer) {
    char alt[NAME_LEN];
    snprintf(alt, sizeof alt, "%s", arg);
    char *save = NULL;
    for (char *a = strtok_r(alt, "|", &save); a; a = strtok_r(NULL, "|", &save)) {
        char name[NAME_LEN], *t = trim(a), *o = name;
        for (; *t && o < name + NAME_LEN - 8; ++t) {
            if (t[0] == '{' && t[1] == 'i' && t[2] == '}') {
                o += snprintf(o, 8, "%d", layer);
                t += 2;
            } else {
                *o++ = *t;
            }
        }
        *o = 0;
        tensor_t *tt = tensor_find(m, name);
        if (tt) return tt;
    }
    return NULL;
}

/* ------------------------------------------------------------------------------------------ */
/* The op interpreter: one line of the definition, as "Local inference and architectures",    */
/* section "The operations", defines each op (embed, rms_norm, matmul, add_bias, norm_heads,    */
/* rope, attention, add, mul, silu, gelu, gelu_tanh, relu, scale, copy, last), and section      */
/* "Rules" its operands: `a | b` takes the first tensor present, {i} is the layer index.       */
/* ------------------------------------------------------------------------------------------ */
static int run_step(orc_model *m, const step_t *st, int layer, const int32_t *tokens, int n,
                    int64_t pos) {
    const char *op = st->op;
    /* source register: first argument (in-place form: the destination itself) */
    reg_t *src = st->nargs > 0 ? reg_find(m, st->args[0]) : NULL;

    if (!strcmp(op, "embed")) {
        tensor_t *T = tensor_arg(m, st->args[0], layer);
        if (!T) return fail(m, "line %d: missing tensor %s", st->line, st->args[0]);
        int64_t w = T->ne[0];
        float *tmp = (float *)malloc(sizeof(float) * (size_t)w);
        reg_t *d = reg_set(m, st->dst, n, (int)w);
        for (int r = 0; r < n; ++r) {
            if (tokens[r] < 0 || tokens[r] >= T->ne[1]) { free(tmp); return fail(m, "token out of range"); }
            dequant_row(T->type, T->data + row_bytes(T->type, w) * (size_t)tokens[r], w, tmp);
            memcpy(d->v + (size_t)r * w, tmp, sizeof(float) * (size_t)w);
        }
        free(tmp);
        return ORC_OK;
    }
    if (!src) return fail(m, "line %d: register %s is not set", st->line, st->nargs ? st->args[0] : "?");
    int rows = src->rows, width = src->width;

    if (!strcmp(op, "matmul")) {
        /* y[r][j] = sum_k W[j][k] * src[r][k]; W stored with ne[0] = k (in-features) contiguous */
        tensor_t *W = tensor_arg(m, st->args[1], layer);
        if (!W) return fail(m, "line %d: missing tensor %s", st->line, st->args[1]);
        if (W->ne[0] != width) return fail(m, "line %d: shape mismatch %s", st->line, W->name);
        int64_t K = W->ne[0], N = W->ne[1];
        float *out = (float *)malloc(sizeof(float) * (size_t)rows * N);
        size_t rb = row_bytes(W->type, K);
#pragma omp parallel
        {
            float *wrow = (float *)malloc(sizeof(float) * (size_t)K);
#pragma omp for schedule(static)
            for (int64_t j = 0; j < N; ++j) {
                dequant_row(W->type, W->data + rb * (size_t)j, K, wrow);
                for (int r = 0; r < rows; ++r) {
                    const float *x = src->v + (size_t)r * K;
                    double acc = 0.0;
                    for (int64_t k = 0; k < K; ++k) acc += (double)wrow[k] * (double)x[k];
                    out[(size_t)r * N + j] = (float)acc;
                }
            }
            free(wrow);
        }
        reg_t *d = reg_set(m, st->dst, rows, (int)N);
        memcpy(d->v, out, sizeof(float) * (size_t)rows * N);
        free(out);
        return ORC_OK;
    }

    /* everything else keeps the shape; compute into a fresh buffer, then store */
    float *y = (float *)malloc(sizeof(float) * (size_t)rows * width);
    memcpy(y, src->v, sizeof(float) * (size_t)rows * width);
    int out_rows = rows;

    if (!strcmp(op, "rms_norm")) {
        tensor_t *w = tensor_arg(m, st->args[1], layer);
        if (!w || w->type != T_F32 || w->ne[0] != width) { free(y); return fail(m, "line %d: bad norm weight", st->line); }
        for (int r = 0; r < rows; ++r)
            rms_norm_vec(src->v + (size_t)r * width, (const float *)w->data, width, m->eps, y + (size_t)r * width);
    } else if (!strcmp(op, "add_bias")) {
        tensor_t *b = tensor_arg(m, st->args[1], layer);
        if (!b || b->type != T_F32 || b->ne[0] != width) { free(y); return fail(m, "line %d: bad bias", st->line); }
        for (int r = 0; r < rows; ++r)
            for (int j = 0; j < width; ++j) y[(size_t)r * width + j] += ((const float *)b->data)[j];
    } else if (!strcmp(op, "norm_heads")) {
        /* per-head RMSNorm over head_dim with a weight of length head_dim */
        tensor_t *w = tensor_arg(m, st->args[1], layer);
        const char *cnt = meta_arch(m, st->args[2]);
        if (!w || !cnt) { free(y); return fail(m, "line %d: bad norm_heads", st->line); }
        int nh = atoi(cnt), hd = width / nh;
        if (w->ne[0] != hd || hd * nh != width) { free(y); return fail(m, "line %d: norm_heads shape", st->line); }
        for (int r = 0; r < rows; ++r)
            for (int h = 0; h < nh; ++h)
                rms_norm_vec(src->v + (size_t)r * width + h * hd, (const float *)w->data, hd, m->eps,
                             y + (size_t)r * width + h * hd);
    } else if (!strcmp(op, "rope")) {
        const char *cnt = meta_arch(m, st->args[1]);
        if (!cnt) { free(y); return fail(m, "line %d: bad rope", st->line); }
        int nh = atoi(cnt), hd = width / nh;
        for (int r = 0; r < rows; ++r)
            for (int h = 0; h < nh; ++h)
                rope_head(y + (size_t)r * width + h * hd, hd, pos + r, m->rope_base, m->rope_adjacent);
    } else if (!strcmp(op, "attention")) {
        /*
         * Append this call's K and V rows at positions pos .. pos+rows-1, then for every row r
         * (absolute position p = pos + r) attend causally over the cache: keys t <= p, and on a
         * sliding-window layer only t > p - window. Q head h reads KV head h / (n_head/n_head_kv).
         */
        reg_t *kr = reg_find(m, st->args[1]), *vr = reg_find(m, st->args[2]);
        if (layer < 0 || !kr || !vr) { free(y); return fail(m, "line %d: attention needs q, k, v in a block", st->line); }
        int hd = m->head_dim, nkv = m->n_head_kv, nh = width / hd, grp = nh / nkv;
        if (kr->width != nkv * hd || vr->width != nkv * hd || nh * hd != width) { free(y); return fail(m, "line %d: attention shapes", st->line); }
        if (pos + rows > m->max_ctx) { free(y); return fail(m, "context full"); }
        for (int r = 0; r < rows; ++r)
            for (int g = 0; g < nkv; ++g) {
                float *kd = m->K[layer] + ((size_t)g * m->max_ctx + pos + r) * hd;
                float *vd = m->V[layer] + ((size_t)g * m->max_ctx + pos + r) * hd;
                const float *ks = kr->v + (size_t)r * kr->width + g * hd, *vs = vr->v + (size_t)r * vr->width + g * hd;
                for (int i = 0; i < hd; ++i) {
                    kd[i] = m->kv_f16 ? round_to_half(ks[i]) : ks[i];
                    vd[i] = m->kv_f16 ? round_to_half(vs[i]) : vs[i];
                }
            }
        int windowed = m->window > 0 && !(m->window_pattern > 0 && layer % m->window_pattern == m->window_pattern - 1);
        for (int r = 0; r < rows; ++r) {
            int64_t p = pos + r;
            int64_t t0 = windowed && p - m->window + 1 > 0 ? p - m->window + 1 : 0;
            for (int h = 0; h < nh; ++h) {
                int g = h / grp;
                attend_head(src->v + (size_t)r * width + h * hd, m->K[layer] + (size_t)g * m->max_ctx * hd,
                            m->V[layer] + (size_t)g * m->max_ctx * hd, hd, t0, p, y + (size_t)r * width + h * hd);
            }
        }
    } else if (!strcmp(op, "silu") || !strcmp(op, "gelu") || !strcmp(op, "gelu_tanh") || !strcmp(op, "relu")) {
        double (*f)(double) = !strcmp(op, "silu") ? op_silu : !strcmp(op, "gelu") ? op_gelu
                            : !strcmp(op, "gelu_tanh") ? op_gelu_tanh : op_relu;
        for (size_t i = 0; i < (size_t)rows * width; ++i) y[i] = (float)f((double)y[i]);
    } else if (!strcmp(op, "mul") || !strcmp(op, "add")) {
        reg_t *b = st->nargs > 1 ? reg_find(m, st->args[1]) : NULL;
        if (!b || b->rows != rows || b->width != width) { free(y); return fail(m, "line %d: %s shapes", st->line, op); }
        int mul = !strcmp(op, "mul");
        for (size_t i = 0; i < (size_t)rows * width; ++i) y[i] = mul ? y[i] * b->v[i] : y[i] + b->v[i];
    } else if (!strcmp(op, "scale")) {
        const char *lit = st->nargs > 1 ? st->args[1] : NULL;
        const char *mv = lit ? meta_arch(m, lit) : NULL;
        float c = (float)atof(mv ? mv : lit ? lit : "1");
        for (size_t i = 0; i < (size_t)rows * width; ++i) y[i] = y[i] * c;
    } else if (!strcmp(op, "copy")) {
        /* y already holds the source */
    } else if (!strcmp(op, "last")) {
        memmove(y, y + (size_t)(rows - 1) * width, sizeof(float) * width);
        out_rows = 1;
    } else {
        free(y);
        return fail(m, "line %d: unsupported op %s", st->line, op);
    }
    reg_t *d = reg_set(m, st->dst, out_rows, width);
    memcpy(d->v, y, sizeof(float) * (size_t)out_rows * width);
    free(y);
    return ORC_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* Public entry points (called through ctypes by the tests)                                    */
/* ------------------------------------------------------------------------------------------ */
const char *orc_last_error(orc_model *m) { return m ? m->err : "null model"; }

/* metadata: "key=value\n" lines (GGUF metadata keys) */
orc_model *orc_create(const char *file_arch, const char *archdef, const char *metadata, int64_t max_ctx,
                      char *err, int errlen) {
    orc_model *m = (orc_model *)calloc(1, sizeof(orc_model));
    char *md = strdup(metadata), *save = NULL;
    for (char *l = strtok_r(md, "\n", &save); l && m->n_meta < MAX_META; l = strtok_r(NULL, "\n", &save)) {
        char *eq = strchr(l, '=');
        if (!eq) continue;
        *eq = 0;
        snprintf(m->meta_k[m->n_meta], 96, "%s", trim(l));
        snprintf(m->meta_v[m->n_meta], 64, "%s", trim(eq + 1));
        ++m->n_meta;
    }
    free(md);
    if (parse_archdef(m, file_arch, archdef) != ORC_OK) goto bad;
    const char *v;
#define NEED(field, name, conv)                                                  \
    if (!(v = meta_arch(m, name))) { fail(m, "missing metadata %s.%s", m->arch, name); goto bad; } \
    m->field = conv(v);
    NEED(n_layer, "block_count", atoi)
    NEED(n_embd, "embedding_length", atoi)
    NEED(n_head, "head_count", atoi)
    NEED(n_head_kv, "head_count_kv", atoi)
    NEED(eps, "layer_norm_rms_epsilon", atof)
    NEED(rope_base, "freq_base", atof)
#undef NEED
    v = meta_arch(m, "key_length");
    m->head_dim = v ? atoi(v) : m->n_embd / m->n_head;
    v = meta_arch(m, "sliding_window");
    m->window = v ? atoi(v) : 0;
    m->max_ctx = max_ctx;
    m->K = (float **)calloc((size_t)m->n_layer, sizeof(float *));
    m->V = (float **)calloc((size_t)m->n_layer, sizeof(float *));
    for (int l = 0; l < m->n_layer; ++l) {
        m->K[l] = (float *)calloc((size_t)m->n_head_kv * max_ctx * m->head_dim, sizeof(float));
        m->V[l] = (float *)calloc((size_t)m->n_head_kv * max_ctx * m->head_dim, sizeof(float));
        if (!m->K[l] || !m->V[l]) { fail(m, "out of memory for the KV cache"); goto bad; }
    }
    return m;
bad:
    if (err && errlen > 0) snprintf(err, (size_t)errlen, "%s", m->err);
    /* partial model: the caller only reads err */
    return NULL;
}

int orc_add_tensor(orc_model *m, const char *name, int type, const int64_t *ne, int ndims, const void *data,
                   size_t nbytes) {
    if (ndims < 1 || ndims > 4) return fail(m, "bad ndims for %s", name);
    if (type != T_F32 && type != T_F16 && type != T_Q8_0 && type != T_Q4_0) return fail(m, "bad type for %s", name);
    if ((type == T_Q8_0 || type == T_Q4_0) && ne[0] % 32) return fail(m, "%s: row not a whole number of blocks", name);
    size_t want = row_bytes(type, ne[0]);
    for (int i = 1; i < ndims; ++i) want *= (size_t)ne[i];
    if (want != nbytes) return fail(m, "%s: %zu bytes, expected %zu", name, nbytes, want);
    if (m->n_tensors == m->cap_tensors) {
        m->cap_tensors = m->cap_tensors ? 2 * m->cap_tensors : 64;
        m->tensors = (tensor_t *)realloc(m->tensors, sizeof(tensor_t) * (size_t)m->cap_tensors);
    }
    tensor_t *t = tensor_find(m, name);
    if (!t) t = &m->tensors[m->n_tensors++];
    memset(t, 0, sizeof *t);
    snprintf(t->name, sizeof t->name, "%s", name);
    t->type = type;
    t->ndims = ndims;
    for (int i = 0; i < 4; ++i) t->ne[i] = i < ndims ? ne[i] : 1;
    t->data = (const uint8_t *)data;
    return ORC_OK;
}

int orc_reset_kv(orc_model *m) {
    m->kv_len = 0;
    return ORC_OK;
}

/* Write n positions [pos0, pos0+n) of layer's cache: k, v laid out [n_head_kv][n][head_dim]. */
int orc_write_kv(orc_model *m, int layer, int64_t pos0, int64_t n, const float *k, const float *v) {
    if (layer < 0 || layer >= m->n_layer || pos0 < 0 || pos0 + n > m->max_ctx) return fail(m, "bad kv range");
    int hd = m->head_dim;
    for (int g = 0; g < m->n_head_kv; ++g) {
        float *kd = m->K[layer] + ((size_t)g * m->max_ctx + pos0) * hd, *vd = m->V[layer] + ((size_t)g * m->max_ctx + pos0) * hd;
        const float *ks = k + (size_t)g * n * hd, *vs = v + (size_t)g * n * hd;
        for (int64_t i = 0; i < n * hd; ++i) {
            kd[i] = m->kv_f16 ? round_to_half(ks[i]) : ks[i];
            vd[i] = m->kv_f16 ? round_to_half(vs[i]) : vs[i];
        }
    }
    return ORC_OK;
}

/* Store keys and values rounded to f16 from now on (on != 0); call before the first forward. */
int orc_set_kv_f16(orc_model *m, int on) {
    m->kv_f16 = on != 0;
    return ORC_OK;
}

/* Read positions [pos0, pos0+n) of layer's cache into k, v laid out [n_head_kv][n][head_dim]. */
int orc_read_kv(orc_model *m, int layer, int64_t pos0, int64_t n, float *k, float *v) {
    if (layer < 0 || layer >= m->n_layer || pos0 < 0 || pos0 + n > m->max_ctx) return fail(m, "bad kv range");
    int hd = m->head_dim;
    for (int g = 0; g < m->n_head_kv; ++g) {
        memcpy(k + (size_t)g * n * hd, m->K[layer] + ((size_t)g * m->max_ctx + pos0) * hd, sizeof(float) * n * hd);
        memcpy(v + (size_t)g * n * hd, m->V[layer] + ((size_t)g * m->max_ctx + pos0) * hd, sizeof(float) * n * hd);
    }
    return ORC_OK;
}

int orc_set_kv_len(orc_model *m, int64_t len) {
    if (len < 0 || len > m->max_ctx) return fail(m, "bad kv length");
    m->kv_len = len;
    return ORC_OK;
}

/*
 * Run the forward over n tokens starting at absolute position pos (pos must equal the number of
 * positions already in the cache). Writes the last row of register `logits` (vocab floats) and,
 * when x_out is not NULL, the last row of register x after the epilogue.
 * layer_x (optional): the last row of x after each block, [n_layer][n_embd].
 */
int orc_forward(orc_model *m, const int32_t *tokens, int n, int64_t pos, float *logits, float *x_out,
                float *layer_x) {
    if (n < 1) return fail(m, "n must be >= 1");
    if (pos != m->kv_len) return fail(m, "pos %lld != kv length %lld", (long long)pos, (long long)m->kv_len);
    if (pos + n > m->max_ctx) return fail(m, "context full");
    for (int s = 0; s < m->n_steps[0]; ++s)
        if (run_step(m, &m->steps[0][s], -1, tokens, n, pos)) return ORC_ERR;
    for (int l = 0; l < m->n_layer; ++l) {
        for (int s = 0; s < m->n_steps[1]; ++s)
            if (run_step(m, &m->steps[1][s], l, tokens, n, pos)) return ORC_ERR;
        if (layer_x) {
            reg_t *x = reg_find(m, "x");
            if (x) memcpy(layer_x + (size_t)l * x->width, x->v + (size_t)(x->rows - 1) * x->width, sizeof(float) * x->width);
        }
    }
    for (int s = 0; s < m->n_steps[2]; ++s)
        if (run_step(m, &m->steps[2][s], -1, tokens, n, pos)) return ORC_ERR;
    m->kv_len = pos + n;
    reg_t *lg = reg_find(m, "logits");
    if (!lg) return fail(m, "no logits register");
    memcpy(logits, lg->v + (size_t)(lg->rows - 1) * lg->width, sizeof(float) * lg->width);
    if (x_out) {
        reg_t *x = reg_find(m, "x");
        memcpy(x_out, x->v + (size_t)(x->rows - 1) * x->width, sizeof(float) * x->width);
    }
    return ORC_OK;
}

int orc_steps(orc_model *m, int section) { return section >= 0 && section < 3 ? m->n_steps[section] : -1; }
int orc_head_dim(orc_model *m) { return m->head_dim; }
int orc_rope_adjacent(orc_model *m) { return m->rope_adjacent; }
int orc_window_pattern(orc_model *m) { return m->window_pattern; }

void orc_destroy(orc_model *m) {
    if (!m) return;
    for (int i = 0; i < m->n_regs; ++i) free(m->regs[i].v);
    if (m->K)
        for (int l = 0; l < m->n_layer; ++l) { free(m->K[l]); free(m->V[l]); }
    free(m->K);
    free(m->V);
    free(m->tensors);
    free(m);
}

/* ---- single ops, for the tests that pin each op against its closed form ----------------- */
void orc_dequant(int type, const void *row, int64_t k, float *out) { dequant_row(type, (const uint8_t *)row, k, out); }
float orc_half_to_float(uint16_t h) { return half_to_float(h); }
float orc_round_to_half(float f) { return round_to_half(f); }

void orc_rms_norm(const float *x, const float *w, int n, double eps, float *y) { rms_norm_vec(x, w, n, eps, y); }

void orc_rope(float *v, int n_heads, int hd, int64_t pos, double base, int adjacent) {
    for (int h = 0; h < n_heads; ++h) rope_head(v + (size_t)h * hd, hd, pos, base, adjacent);
}

/* q: [hd]; K, V: [n][hd]; attends over rows t0..t1 */
void orc_attend(const float *q, const float *K, const float *V, int hd, int64_t t0, int64_t t1, float *o) {
    attend_head(q, K, V, hd, t0, t1, o);
}

/* kind: 0 silu, 1 gelu, 2 gelu_tanh, 3 relu */
void orc_act(int kind, const float *x, int64_t n, float *y) {
    for (int64_t i = 0; i < n; ++i) {
        double v = x[i];
        y[i] = (float)(kind == 0 ? op_silu(v) : kind == 1 ? op_gelu(v) : kind == 2 ? op_gelu_tanh(v) : op_relu(v));
    }
}

/* y[j] = sum_k W[j][k] x[k] for a GGUF tensor with ne = {k, n} */
void orc_matvec(int type, const void *W, int64_t k, int64_t n, const float *x, float *y) {
    size_t rb = row_bytes(type, k);
    float *wrow = (float *)malloc(sizeof(float) * (size_t)k);
    for (int64_t j = 0; j < n; ++j) {
        dequant_row(type, (const uint8_t *)W + rb * (size_t)j, k, wrow);
        double acc = 0.0;
        for (int64_t i = 0; i < k; ++i) acc += (double)wrow[i] * (double)x[i];
        y[j] = (float)acc;
    }
    free(wrow);
}
