// k_stream.cuh -- the persistent streaming decode-step kernel: one forward at n = 1 ("Execution
// contract", section "Forward phase") as a single cooperative launch with one CTA per SM.
//
// A decode step at batch size 1 reads every weight once and the KV cache over the allowed keys
// once; it is bound by HBM. Launched as one kernel per fused node, every kernel boundary costs the
// launch ramp, the staging of the input vector and the spread of CTA end times, during which HBM
// idles. Here the fused plan's nodes become phases of one kernel, and the data that does not depend
// on the step's earlier phases -- weight rows, and the KV rows of earlier positions -- is streamed
// by a producer warp per CTA that never waits for a phase to finish:
//
//   producer warp  one thread walks the CTA's share of every phase in order (GEMV row tiles, the
//                  key tiles of its attention slices) and bulk-copies them (cp.async.bulk, TMA)
//                  into a ring of 32 KB shared-memory slots, each completing on an mbarrier; it
//                  only waits for a slot to be released. With 4-8 slots (128-256 KB per SM) it runs
//                  up to that far ahead of the consumers, across phase boundaries.
//   8 consumer     run the phases in order. Before a phase they wait until every CTA has finished
//   warps          the previous one (a grid-wide arrival counter, release / acquire), then stage the
//                  phase's input and consume the ring tiles as they land.
//
// GEMV phases (`matmul`, with the folded rms_norm prologue, bias, residual-add and act(gate) * up
// epilogues of "Local inference and architectures", section "The format"): each CTA takes a
// contiguous, balanced range of the phase's rows; a tile is one or two slots of whole rows. The
// thread that owns 32-byte chunk c of a row reads it from the slot (two 16-byte shared loads, in a
// lane-dependent order that keeps them free of bank conflicts) for every row of the tile it
// handles, with the matching x values loaded once per tile into registers; codes become floats
// without conversion instructions (a byte in the mantissa of 2^23) and products accumulate with
// packed f32x2 FMAs, all in f32 ("we multiply in f32", section "Choosing the engine"). Partial
// sums meet through a warp reduce-scatter and one shared-memory exchange per tile.
//
// Attention phases (`attention` with the per-head transforms and the KV append folded in): the
// split count follows the context length; the key tiles of the CTA's slices are streamed as K
// slots and V slots; the new position's key and value are appended by the CTA whose slice holds
// that position and enter its softmax from registers (the producer never copies a row this step
// writes). The slices are merged by the last CTA of each KV head (attn_dev.cuh).
//
// Small phases (embed, rms_norm with residual, elementwise ops, per-head transforms, copies, the
// greedy argmax that advances the position) run on the consumer threads spread over the CTAs.
//
// Every wait is bounded by wall-clock time (1 s on the ring, 2 s for the previous phase). A wait that
// runs out sets ERR_STREAM (ERR_BARRIER for the grid-wide count)
// in the device state and an abort flag in the CTA: the consumers then run to the end of the
// phase list without waiting (they still arrive at the grid counter, so other CTAs do not wait for
// them), the producer stops issuing and waits, with the full bound, for its copies still in flight,
// and every thread meets at a final block barrier before the CTA exits.
#pragma once

#include "async_dev.cuh"
#include "attn_dev.cuh"
#include "gemv_dev.cuh"
#include "misc_dev.cuh"

namespace syn {

constexpr int kStreamWarps = kConsumerThreads / 32;           // consumer warps
constexpr int kStreamThreads = kConsumerThreads + 32;         // + the producer warp
constexpr int kMaxSlots = 8;
constexpr int kRM = 8;                                       // GEMV tile rows per consumer thread
constexpr unsigned long long kWaitNs = 1000000000ull;         // a ring wait gives up after 1 s
constexpr unsigned long long kGridWaitNs = 2000000000ull;     // the wait for the previous phase, 2 s

SYN_DEV unsigned long long stream_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
SYN_DEV unsigned ld_acquire_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
SYN_DEV void red_release_add_u32(unsigned *p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
SYN_DEV uint4 lds128(const uint8_t *p) { return *reinterpret_cast<const uint4 *>(p); }

// Bounded wait for phase `par` of mbarrier `bar`: `spin` < 0 bounds it by wall-clock time (kWaitNs),
// else by that many polls (0: give up at once; test support). Returns false when it gave up or when
// `abort` was raised meanwhile.
SYN_DEV bool stream_wait(uint64_t *bar, unsigned par, int spin, volatile int *abort) {
    if (spin >= 0) {
        for (int i = 0; i < spin; ++i)
            if (mbar_try(bar, par)) return true;
        return false;
    }
    const unsigned long long deadline = stream_ns() + kWaitNs;
    for (unsigned i = 1;; ++i) {
        if (mbar_try(bar, par)) return true;
        if ((i & 15u) == 0) {
            if (*abort) return false;
            if (stream_ns() > deadline) return false;
        }
    }
}

// ------------------------------------------------------------------------------- GEMV tiling
// The tiles of one CTA, in order: rows [v, v + n) of the phase's row list (pairs for gate/up)
// within segment `seg`, row0 the first row inside that segment.
struct GemvTiles {
    int v, v1, cap;
    SYN_DEV GemvTiles(const StreamGemv &g, bool gate_up, int cta, int ncta) {
        v = (int)((int64_t)g.rows * cta / ncta);
        v1 = (int)((int64_t)g.rows * (cta + 1) / ncta);
        cap = g.slots * (gate_up ? g.rs / 2 : g.rs);
    }
    // next tile; false when the range is done
    SYN_DEV bool next(const StreamGemv &g, int &seg, int &row0, int &n) {
        if (v >= v1) return false;
        seg = (v >= g.seg_end[0]) + (v >= g.seg_end[1]);
        const int s0 = seg == 0 ? 0 : g.seg_end[seg - 1];
        n = min(cap, min(v1 - v, g.seg_end[seg] - v));
        row0 = v - s0;
        v += n;
        return true;
    }
};
SYN_DEV int gemv_tile_slots(const StreamGemv &g, bool gate_up, int n) {
    const int per = gate_up ? g.rs / 2 : g.rs;
    return (n + per - 1) / per;
}

// ------------------------------------------------------------------------------- attention split
// Slices per KV head at this step: about two key tiles or more per slice, at most `smax` (so that
// KV heads x slices fill the SMs once at long context).
SYN_DEV int stream_splits(int len, int smax, int tk) {
    const int s = (len + 2 * tk - 1) / (2 * tk);
    return max(1, min(smax, s));
}
SYN_DEV void stream_attn_range(const AttnParams &a, int pos, int S, int split, int &start, int &end) {
    const int lo = a.window > 0 ? max(0, pos - a.window + 1) : 0;
    const int len = pos - lo + 1;
    const int chunk = (len + S - 1) / S;
    start = lo + split * chunk;
    end = min(pos + 1, start + chunk);
}

// ------------------------------------------------------------------------------- producer
template <int HD, int GP>
SYN_DEV void stream_producer(const StreamParams &sp, uint8_t *ring, uint64_t *full, uint64_t *empty, int pos,
                             volatile int *abort) {
    const int cta = blockIdx.x, ncta = gridDim.x, NS = sp.nslots;
    int *err = &sp.state->err;
    int u = 0;   // slot uses issued
    // the slot of use u once its previous use was released; nullptr when the wait gave up or the
    // consumers aborted
    auto claim = [&](uint64_t *&bar) -> uint8_t * {
        const int s = u % NS;
        if (u >= NS) {
            const unsigned par = (unsigned)((u / NS) - 1) & 1u;
            const bool got = stream_wait(&empty[s], par, sp.spin, abort);
            if (!got) {
                if (!*abort) atomicOr(err, ERR_STREAM);
                *abort = 1;
                return nullptr;
            }
        }
        if (*abort) return nullptr;
        bar = &full[s];
        return ring + (size_t)s * kSlotBytes;
    };
    bool ok = true;
    for (int ph = 0; ph < sp.nphases && ok; ++ph) {
        const PhaseDesc &d = sp.phases[ph];
        const int kind = d.kind;
        if (kind == PH_GEMV) {
            const GemvParams &p = d.gemv;
            const StreamGemv &g = d.sg;
            const bool gu = p.gate_up != 0;
            const size_t rb = (size_t)p.seg[0].W.row_bytes;
            const int ss = (int)p.seg[0].W.scale_stride;
            const bool q = p.seg[0].W.scales != nullptr;
            GemvTiles T(g, gu, cta, ncta);
            int seg, row0, n;
            while (ok && T.next(g, seg, row0, n)) {
                const int nsl = gemv_tile_slots(g, gu, n);
                for (int k = 0; k < nsl; ++k) {
                    uint64_t *bar;
                    uint8_t *dst = claim(bar);
                    if (!dst) { ok = false; break; }
                    if (!gu) {
                        const DevMatrix &W = p.seg[seg].W;
                        const int r = row0 + k * g.rs, cnt = min(g.rs, n - k * g.rs);
                        const unsigned cb = (unsigned)(cnt * rb), sb = q ? (unsigned)(cnt * ss * 2) : 0u;
                        mbar_expect_tx(bar, cb + sb);
                        bulk_g2s(dst, static_cast<const uint8_t *>(W.codes) + (size_t)r * rb, cb, bar);
                        if (q) bulk_g2s(dst + (size_t)g.rs * rb, W.scales + (size_t)r * ss, sb, bar);
                    } else {
                        const int h = g.rs / 2;
                        const int r = row0 + k * h, cnt = min(h, n - k * h);
                        const unsigned cb = (unsigned)(cnt * rb), sb = q ? (unsigned)(cnt * ss * 2) : 0u;
                        mbar_expect_tx(bar, 2 * (cb + sb));
                        bulk_g2s(dst, static_cast<const uint8_t *>(p.seg[0].W.codes) + (size_t)r * rb, cb, bar);
                        bulk_g2s(dst + (size_t)h * rb, static_cast<const uint8_t *>(p.seg[1].W.codes) + (size_t)r * rb, cb, bar);
                        if (q) {
                            uint8_t *sd = dst + (size_t)g.rs * rb;
                            bulk_g2s(sd, p.seg[0].W.scales + (size_t)r * ss, sb, bar);
                            bulk_g2s(sd + (size_t)h * ss * 2, p.seg[1].W.scales + (size_t)r * ss, sb, bar);
                        }
                    }
                    ++u;
                }
            }
        } else if (kind == PH_ATTN) {
            const AttnParams &a = d.attn;
            constexpr int TK = kAttnWarps * AttnShape<HD, GP>::KB;
            const int es = a.kv_f16 ? 2 : 4;
            const int lo = a.window > 0 ? max(0, pos - a.window + 1) : 0;
            const int S = stream_splits(pos - lo + 1, a.splits, TK);
            for (int unit = cta; ok && unit < a.n_kv * S; unit += ncta) {
                const int gh = unit % a.n_kv, split = unit / a.n_kv;
                int start, end;
                stream_attn_range(a, pos, S, split, start, end);
                const int old_end = min(end, pos);
                const uint8_t *Kg = static_cast<const uint8_t *>(a.kcache) + (size_t)gh * a.max_ctx * HD * es;
                const uint8_t *Vg = static_cast<const uint8_t *>(a.vcache) + (size_t)gh * a.max_ctx * HD * es;
                for (int t0 = start; ok && t0 < old_end; t0 += TK) {
                    const unsigned bytes = (unsigned)(min(TK, old_end - t0) * HD * es);
                    for (int kv = 0; kv < 2; ++kv) {
                        uint64_t *bar;
                        uint8_t *dst = claim(bar);
                        if (!dst) { ok = false; break; }
                        mbar_expect_tx(bar, bytes);
                        bulk_g2s(dst, (kv ? Vg : Kg) + (size_t)t0 * HD * es, bytes, bar);
                        ++u;
                    }
                }
            }
        }
    }
    // no copy may land in shared memory after the CTA has left: wait (wall-clock bound, whatever the
    // test setting) for the copies of the last uses
    volatile int no_abort = 0;
    for (int v = max(0, u - NS); v < u; ++v)
        if (!stream_wait(&full[v % NS], (unsigned)(v / NS) & 1u, -1, &no_abort)) atomicOr(err, ERR_STREAM);
}

// ------------------------------------------------------------------------------- consumers
struct StreamCons {
    uint8_t *ring;
    float *aux;
    uint64_t *full, *empty;
    volatile int *abort;
    int *err;
    int NS;
    int u;          // slot uses consumed
    int spin;       // wait bound (see stream_wait)
    float *red;     // [2][kStreamWarps][kRM]
    float *sred;    // 32 floats
    int buf;
    // wait for use u + k of the ring (all lanes of the calling warp poll); false once aborted
    SYN_DEV bool wait_full(int k) {
        const int v = u + k;
        if (*abort) return false;
        if (stream_wait(&full[v % NS], (unsigned)(v / NS) & 1u, spin, abort)) return true;
        if (!*abort) atomicOr(err, ERR_STREAM);
        *abort = 1;
        return false;
    }
    SYN_DEV uint8_t *slot(int k) const { return ring + (size_t)((u + k) % NS) * kSlotBytes; }
    // this warp is done reading uses u .. u + n - 1
    SYN_DEV void release(int n) {
        __syncwarp();
        if ((threadIdx.x & 31) == 0)
            for (int k = 0; k < n; ++k) mbar_arrive(&empty[(u + k) % NS]);
        u += n;
    }
};

// 16 code bytes . x values (the chunk halves): Q8_0 offset-binary bytes, Q4_0 one block (low
// nibbles: elements 0..15, high nibbles: 16..31), f16 halves, f32 floats.
SYN_DEV float dot16_q8(const uint4 c, const float *x) {
    float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
    const float2 bias = make_float2(-8388736.f, -8388736.f);   // 2^23 + 128
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 q01 = __fadd2_rn(make_float2(magic(w[i], 0), magic(w[i], 1)), bias);
        const float2 q23 = __fadd2_rn(make_float2(magic(w[i], 2), magic(w[i], 3)), bias);
        a0 = __ffma2_rn(q01, make_float2(x[4 * i], x[4 * i + 1]), a0);
        a1 = __ffma2_rn(q23, make_float2(x[4 * i + 2], x[4 * i + 3]), a1);
    }
    return (a0.x + a0.y) + (a1.x + a1.y);
}
SYN_DEV float dot16_q4(const uint4 c, const float *x) {
    float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
    const float2 bias = make_float2(-8388616.f, -8388616.f);   // 2^23 + 8
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = w[i] & 0x0F0F0F0Fu, hi = (w[i] >> 4) & 0x0F0F0F0Fu;
        a0 = __ffma2_rn(__fadd2_rn(make_float2(magic(lo, 0), magic(lo, 1)), bias), make_float2(x[4 * i], x[4 * i + 1]), a0);
        a1 = __ffma2_rn(__fadd2_rn(make_float2(magic(lo, 2), magic(lo, 3)), bias), make_float2(x[4 * i + 2], x[4 * i + 3]), a1);
        a0 = __ffma2_rn(__fadd2_rn(make_float2(magic(hi, 0), magic(hi, 1)), bias), make_float2(x[16 + 4 * i], x[17 + 4 * i]), a0);
        a1 = __ffma2_rn(__fadd2_rn(make_float2(magic(hi, 2), magic(hi, 3)), bias), make_float2(x[18 + 4 * i], x[19 + 4 * i]), a1);
    }
    return (a0.x + a0.y) + (a1.x + a1.y);
}
SYN_DEV float dot16_f16(const uint4 c, const float *x) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; i += 2) {
        a0 = __ffma2_rn(__half22float2(*reinterpret_cast<const __half2 *>(&w[i])), make_float2(x[2 * i], x[2 * i + 1]), a0);
        a1 = __ffma2_rn(__half22float2(*reinterpret_cast<const __half2 *>(&w[i + 1])), make_float2(x[2 * i + 2], x[2 * i + 3]), a1);
    }
    return (a0.x + a0.y) + (a1.x + a1.y);
}
SYN_DEV float dot16_f32(const uint4 c, const float *x) {
    float2 a = __ffma2_rn(make_float2(__uint_as_float(c.x), __uint_as_float(c.y)), make_float2(x[0], x[1]), make_float2(0.f, 0.f));
    a = __ffma2_rn(make_float2(__uint_as_float(c.z), __uint_as_float(c.w)), make_float2(x[2], x[3]), a);
    return a.x + a.y;
}

// Lane l ends with the warp-wide sum of v[l >> (5 - log2 N)] (N a power of two, at most 32).
template <int N> SYN_DEV float reduce_scatter(float (&v)[N], int lane) {
    int m = 16;
#pragma unroll
    for (int half = N / 2; half >= 1; half >>= 1, m >>= 1) {
        const bool up = lane & m;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = up ? v[i] : v[i + half];
            const float keep = up ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
    }
    float r = v[0];
#pragma unroll
    for (int mm = 16 / N; mm >= 1; mm >>= 1) r += __shfl_xor_sync(0xffffffffu, r, mm);
    return r;
}

template <int WT> struct ChunkShape;
template <> struct ChunkShape<W_Q8_0> { static constexpr int E = 32, SPC = 1; };
template <> struct ChunkShape<W_Q4_0> { static constexpr int E = 64, SPC = 2; };
template <> struct ChunkShape<W_F16> { static constexpr int E = 16, SPC = 0; };
template <> struct ChunkShape<W_F32> { static constexpr int E = 8, SPC = 0; };

template <int WT> SYN_DEV float dot16(const uint4 c, const float *x) {
    if constexpr (WT == W_Q8_0) return dot16_q8(c, x);
    else if constexpr (WT == W_Q4_0) return dot16_q4(c, x);
    else if constexpr (WT == W_F16) return dot16_f16(c, x);
    else return dot16_f32(c, x);
}

// One GEMV phase on the consumer threads.
template <int WT>
SYN_DEV void stream_gemv(const PhaseDesc &d, StreamCons &cs, int cta, int ncta) {
    constexpr int E = ChunkShape<WT>::E, SPC = ChunkShape<WT>::SPC, XH = E / 2;
    const GemvParams &p = d.gemv;
    const StreamGemv &g = d.sg;
    const bool gu = p.gate_up != 0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int K = (int)p.seg[0].W.K;
    const int rb = (int)p.seg[0].W.row_bytes;
    const int ss = (int)p.seg[0].W.scale_stride;
    const int C = g.C;
    float *xs = cs.aux;

    // ---- stage x (times the norm weight), lane-interleaved per 32-chunk slab; sum of squares
    const int slabs = (C + 31) / 32;
    const int n4 = slabs * 32 * E / 4;
    float sq = 0.f;
    for (int base = tid; base < n4; base += 4 * kConsumerThreads) {
        float4 v[4], w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i4 = base + j * kConsumerThreads;
            v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            w[j] = make_float4(1.f, 1.f, 1.f, 1.f);
            if (i4 < n4 && i4 * 4 < K) {
                v[j] = __ldcg(reinterpret_cast<const float4 *>(p.x + i4 * 4));
                if (p.norm_w) w[j] = *reinterpret_cast<const float4 *>(p.norm_w + i4 * 4);
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i4 = base + j * kConsumerThreads;
            if (i4 >= n4) break;
            sq = fmaf(v[j].x, v[j].x, sq);
            sq = fmaf(v[j].y, v[j].y, sq);
            sq = fmaf(v[j].z, v[j].z, sq);
            sq = fmaf(v[j].w, v[j].w, sq);
            *reinterpret_cast<float4 *>(xs + xs_slot<E>(i4 * 4)) =
                make_float4(v[j].x * w[j].x, v[j].y * w[j].y, v[j].z * w[j].z, v[j].w * w[j].w);
        }
    }
    // the block sum's barriers also publish xs to every consumer
    sq = block_sum<ConsumerThreads>(sq, cs.sred);
    const float inv = p.norm_w ? 1.f / sqrtf(sq / (float)K + p.eps) : 1.f;

    // ---- thread -> (row group, chunk) mapping
    const int grp = g.P > 1 ? warp / g.wg : 0;
    const bool active = grp < g.P;
    const int li = g.P > 1 ? (warp - grp * g.wg) * 32 + lane : tid;
    const int cstep = g.P > 1 ? C : kConsumerThreads;    // one chunk per thread when P > 1
    const int h0 = (lane >> 2) & 1;                      // which half of a chunk this lane reads first
    const int hrows = g.rs / 2;

    GemvTiles T(g, gu, cta, ncta);
    int seg, row0, n;
    while (T.next(g, seg, row0, n)) {
        const int nsl = gemv_tile_slots(g, gu, n);
        bool okw = true;
        for (int k = 0; k < nsl; ++k) okw = cs.wait_full(k) && okw;
        // tile position t = k * rs + j (slot k, row j of the slot): present when that row was copied
        auto present = [&](int t) {
            const int k = t / g.rs, j = t - k * g.rs;
            if (k >= nsl) return false;
            if (!gu) return t < n;
            const int hk = min(hrows, n - k * hrows);
            return j < hrows ? j < hk : j - hrows < hk;
        };
        const int R = nsl * g.rs;
        // the epilogue operands of this thread's output row (position tid), fetched before the
        // dot products so that their latency is hidden
        float pre_res = 0.f, pre_b = 0.f, pre_bu = 0.f;
        int out_row = -1;
        if (tid < R && present(tid) && (!gu || (tid % g.rs) < hrows)) {
            const int k = tid / g.rs, j = tid - k * g.rs;
            const GemvSeg &S = p.seg[gu ? 0 : seg];
            out_row = gu ? row0 + k * hrows + j : row0 + tid;
            if (S.epi == EPI_ADD) pre_res = __ldcg(S.out + out_row);
            if (S.bias) pre_b = S.bias[out_row];
            if (gu && p.seg[1].bias) pre_bu = p.seg[1].bias[out_row];
        }
        float acc[kRM];
#pragma unroll
        for (int i = 0; i < kRM; ++i) acc[i] = 0.f;
        if (active && okw) {
            for (int c = li; c < C; c += cstep) {
                // this chunk's x values, the half this lane reads first in xa
                float xa[XH], xb[XH];
                const float *xc = xs + (c >> 5) * 32 * E + (c & 31) * 4;
#pragma unroll
                for (int j = 0; j < XH / 4; ++j) {
                    const float4 a = *reinterpret_cast<const float4 *>(xc + (j + h0 * (XH / 4)) * 128);
                    const float4 b = *reinterpret_cast<const float4 *>(xc + (j + (1 - h0) * (XH / 4)) * 128);
                    xa[4 * j] = a.x; xa[4 * j + 1] = a.y; xa[4 * j + 2] = a.z; xa[4 * j + 3] = a.w;
                    xb[4 * j] = b.x; xb[4 * j + 1] = b.y; xb[4 * j + 2] = b.z; xb[4 * j + 3] = b.w;
                }
#pragma unroll
                for (int i = 0; i < kRM; ++i) {
                    const int t = grp + g.P * i;
                    if (t >= R || !present(t)) continue;
                    const int k = t / g.rs, j = t - k * g.rs;
                    const uint8_t *rowp = cs.slot(k) + (size_t)j * rb + (size_t)c * 32;
                    const uint4 ca = lds128(rowp + h0 * 16), cb = lds128(rowp + (1 - h0) * 16);
                    if constexpr (SPC == 0) {
                        acc[i] += dot16<WT>(ca, xa) + dot16<WT>(cb, xb);
                    } else {
                        const uint16_t *sc = reinterpret_cast<const uint16_t *>(cs.slot(k) + (size_t)g.rs * rb) + (size_t)j * ss;
                        if constexpr (SPC == 1) {
                            acc[i] = fmaf(half_bits_to_float(sc[c]), dot16<WT>(ca, xa) + dot16<WT>(cb, xb), acc[i]);
                        } else {
                            acc[i] = fmaf(half_bits_to_float(sc[2 * c + h0]), dot16<WT>(ca, xa), acc[i]);
                            acc[i] = fmaf(half_bits_to_float(sc[2 * c + 1 - h0]), dot16<WT>(cb, xb), acc[i]);
                        }
                    }
                }
            }
        }
        cs.release(nsl);
        // ---- sums: within the warp (reduce-scatter), then over the warps of the row group
        const float v = reduce_scatter<kRM>(acc, lane);
        float *red = cs.red + cs.buf * kStreamWarps * kRM;
        if ((lane & (32 / kRM - 1)) == 0) red[warp * kRM + lane / (32 / kRM)] = v;
        ConsumerThreads::sync();
        if (out_row >= 0) {
            auto total = [&](int t) {
                const int pg = t % g.P, i = t / g.P;
                float sum = 0.f;
                for (int w = pg * g.wg; w < (pg + 1) * g.wg; ++w) sum += red[w * kRM + i];
                return sum * inv;
            };
            if (gu) {
                const float gv = total(tid) + pre_b, uv = total(tid + hrows) + pre_bu;
                p.seg[0].out[out_row] = apply_act(p.act, gv) * uv;
            } else {
                p.seg[seg].out[out_row] = total(tid) + pre_b + pre_res;
            }
        }
        cs.buf ^= 1;
    }
}

// One attention phase on the consumer threads (decode: one query row at position pos).
template <int HD, int GP, class KV>
SYN_DEV void stream_attn(const PhaseDesc &d, StreamCons &cs, int cta, int ncta, int pos) {
    using Sh = AttnShape<HD, GP>;
    constexpr int EL = Sh::EL, KB = Sh::KB, TK = kAttnWarps * KB;
    const AttnParams &a = d.attn;
    const HeadsParams &h = a.heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.n_head / a.n_kv;
    const int lo = a.window > 0 ? max(0, pos - a.window + 1) : 0;
    const int S = stream_splits(pos - lo + 1, a.splits, TK);
    const float scale = 1.f / sqrtf((float)HD);
    const float2 *rcs = h.rope_cs + (size_t)pos * (HD / 2);
    for (int unit = cta; unit < a.n_kv * S; unit += ncta) {
        const int g = unit % a.n_kv, split = unit / a.n_kv;
        int start, end;
        stream_attn_range(a, pos, S, split, start, end);
        const int old_end = min(end, pos);
        const bool owns_new = start <= pos && pos < end;
        // this warp's copy of the group's query heads
        float q[GP][EL];
        if (a.fuse_heads) {
#pragma unroll
            for (int hq = 0; hq < GP; ++hq) {
                if (hq < G) {
                    const int qh = g * G + hq;
#pragma unroll
                    for (int e = 0; e < EL; ++e) q[hq][e] = __ldcg(h.q + (size_t)qh * HD + lane * EL + e);
                    head_transform<HD>(q[hq], h.bq ? h.bq + (size_t)qh * HD : nullptr, h.wq, h.rope_q, rcs, h.rope_adjacent, h.eps);
                } else {
#pragma unroll
                    for (int e = 0; e < EL; ++e) q[hq][e] = 0.f;
                }
            }
        } else {
            attn_load_q<HD, GP>(a, g, 0, q);
        }
        float m_run = -FLT_MAX, l_run = 0.f;
        float o[GP][EL];
#pragma unroll
        for (int hq = 0; hq < GP; ++hq)
#pragma unroll
            for (int e = 0; e < EL; ++e) o[hq][e] = 0.f;
        if (owns_new && warp == 0) {
            // the new position's key and value: transformed and appended here (folded heads), or
            // already appended by a per-head phase; they enter the softmax from registers
            float kr[KB][EL], vr[KB][EL];
#pragma unroll
            for (int j = 0; j < KB; ++j)
#pragma unroll
                for (int e = 0; e < EL; ++e) { kr[j][e] = 0.f; vr[j][e] = 0.f; }
            KV *kd = static_cast<KV *>(const_cast<void *>(a.kcache)) + ((size_t)g * a.max_ctx + pos) * HD + lane * EL;
            KV *vd = static_cast<KV *>(const_cast<void *>(a.vcache)) + ((size_t)g * a.max_ctx + pos) * HD + lane * EL;
            if (a.fuse_heads) {
#pragma unroll
                for (int e = 0; e < EL; ++e) {
                    kr[0][e] = __ldcg(h.k + (size_t)g * HD + lane * EL + e);
                    vr[0][e] = __ldcg(h.v + (size_t)g * HD + lane * EL + e);
                    if (h.bv) vr[0][e] += h.bv[(size_t)g * HD + lane * EL + e];
                }
                head_transform<HD>(kr[0], h.bk ? h.bk + (size_t)g * HD : nullptr, h.wk, h.rope_k, rcs, h.rope_adjacent, h.eps);
#pragma unroll
                for (int e = 0; e < EL; ++e) {
                    st_kv(kd + e, kr[0][e]);
                    st_kv(vd + e, vr[0][e]);
                }
                // the cache holds the rounded values (f16 cache): attend to what was stored
                if constexpr (sizeof(KV) == 2) {
#pragma unroll
                    for (int e = 0; e < EL; ++e) {
                        kr[0][e] = __half2float(__float2half_rn(kr[0][e]));
                        vr[0][e] = __half2float(__float2half_rn(vr[0][e]));
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < EL; ++e) {
                    if constexpr (sizeof(KV) == 2) {
                        kr[0][e] = __half2float(__ushort_as_half(__ldcg(reinterpret_cast<const unsigned short *>(kd + e))));
                        vr[0][e] = __half2float(__ushort_as_half(__ldcg(reinterpret_cast<const unsigned short *>(vd + e))));
                    } else {
                        kr[0][e] = __ldcg(reinterpret_cast<const float *>(kd + e));
                        vr[0][e] = __ldcg(reinterpret_cast<const float *>(vd + e));
                    }
                }
            }
            attn_step<HD, GP>(q, kr, vr, 1, G, scale, m_run, l_run, o);
        }
        for (int t0 = start; t0 < old_end; t0 += TK) {
            const bool okw = cs.wait_full(0) & cs.wait_full(1);
            const int tw = t0 + warp * KB;
            const int nk = min(KB, old_end - tw);
            if (okw && nk > 0) {
                const KV *sk = reinterpret_cast<const KV *>(cs.slot(0)) + warp * KB * HD + lane * EL;
                const KV *sv = reinterpret_cast<const KV *>(cs.slot(1)) + warp * KB * HD + lane * EL;
                float kr[KB][EL], vr[KB][EL];
#pragma unroll
                for (int j = 0; j < KB; ++j) {
                    if (j < nk) {
                        lds_row<EL>(kr[j], sk + j * HD);
                        lds_row<EL>(vr[j], sv + j * HD);
                    } else {
#pragma unroll
                        for (int e = 0; e < EL; ++e) { kr[j][e] = 0.f; vr[j][e] = 0.f; }
                    }
                }
                attn_step<HD, GP>(q, kr, vr, nk, G, scale, m_run, l_run, o);
            }
            cs.release(2);
        }
        // merge the warps and the slices (the aux region is the merge scratch)
        ConsumerThreads::sync();
        attn_finish<HD, GP>(a, S, g, split, 0, cs.aux, m_run, l_run, o, [] { ConsumerThreads::sync(); });
    }
}

template <int HD, int GP>
SYN_DEV void stream_consumers(const StreamParams &sp, StreamCons &cs, PhaseDesc &d, int pos, float *sv, int *si,
                              int *last, int *flag) {
    const int cta = blockIdx.x, ncta = gridDim.x;
    const bool tr = sp.trace && cta == 0 && threadIdx.x == 0;
    for (int ph = 0; ph < sp.nphases; ++ph) {
        // the phase descriptor into shared memory (every consumer is past the previous phase)
        {
            const int4 *src = reinterpret_cast<const int4 *>(sp.phases + ph);
            int4 *dst = reinterpret_cast<int4 *>(&d);
            for (int i = threadIdx.x; i < (int)(sizeof(PhaseDesc) / 16); i += kConsumerThreads) dst[i] = __ldg(src + i);
        }
        if (tr) sp.trace[3 * ph] = stream_ns();
        if (threadIdx.x == 0) {
            // every CTA has finished phases 0 .. ph-1 (bounded; gives up early once any CTA failed)
            if (ph > 0 && !*cs.abort) {
                const unsigned target = (unsigned)ph * (unsigned)ncta;
                const unsigned long long deadline = stream_ns() + kGridWaitNs;
                for (unsigned i = 1; (int)(ld_acquire_u32(sp.arrivals) - target) < 0; ++i) {
                    if ((i & 63u) == 0) {
                        if (*(volatile int *)cs.err) {   // another CTA gave up: stop waiting
                            *cs.abort = 1;
                            break;
                        }
                        if (stream_ns() > deadline) {
                            atomicOr(cs.err, ERR_BARRIER);
                            *cs.abort = 1;
                            break;
                        }
                    }
                }
            }
            *flag = *cs.abort;
        }
        ConsumerThreads::sync();
        if (tr) sp.trace[3 * ph + 1] = stream_ns();
        const bool run = !*flag;
        switch (d.kind) {
        case PH_GEMV:
            // even when aborted, the tiles are walked (without waiting) to keep the ring accounting
            switch (d.gemv.seg[0].W.wtype) {
            case W_Q8_0: stream_gemv<W_Q8_0>(d, cs, cta, ncta); break;
            case W_Q4_0: stream_gemv<W_Q4_0>(d, cs, cta, ncta); break;
            case W_F16: stream_gemv<W_F16>(d, cs, cta, ncta); break;
            default: stream_gemv<W_F32>(d, cs, cta, ncta); break;
            }
            break;
        case PH_ATTN:
            if (d.attn.kv_f16) stream_attn<HD, GP, __half>(d, cs, cta, ncta, pos);
            else stream_attn<HD, GP, float>(d, cs, cta, ncta, pos);
            break;
        case PH_HEADS:
            if (run) heads_cta<ConsumerThreads>(d.heads, cta, ncta);
            break;
        case PH_EMBED:
            if (run) embed_cta<ConsumerThreads>(d.embed, cta, ncta);
            break;
        case PH_RMS:
            if (run) rms_cta<ConsumerThreads>(d.rms, cta, ncta, cs.sred);
            break;
        case PH_ELT:
            if (run) elt_cta<ConsumerThreads>(d.elt, cta, ncta);
            break;
        case PH_ARGMAX:
            if (run && cta < d.arg_ctas) argmax_cta<ConsumerThreads>(d.argmax, cta, d.arg_ctas, sv, si, last);
            break;
        case PH_COPY:
            if (run)
                for (int i = cta * kConsumerThreads + threadIdx.x; i < d.copy.n; i += ncta * kConsumerThreads)
                    d.copy.dst[i] = __ldcg(d.copy.src + i);
            break;
        }
        // this CTA's writes of the phase are done: count it as arrived
        ConsumerThreads::sync();
        if (threadIdx.x == 0) {
            __threadfence();
            red_release_add_u32(sp.arrivals, 1u);
        }
        if (tr) sp.trace[3 * ph + 2] = stream_ns();
    }
}

// HD, GP: head dimension and padded query-group size of the attention phases (one model has one
// of each); every weight type is handled inside.
template <int HD, int GP>
__global__ void __launch_bounds__(kStreamThreads, 1) k_stream(const StreamParams sp) {
    extern __shared__ uint8_t stream_smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(stream_smem_raw) + 127) & ~uintptr_t(127));
    float *aux = reinterpret_cast<float *>(ring + (size_t)sp.nslots * kSlotBytes);
    __shared__ __align__(8) uint64_t full[kMaxSlots], empty[kMaxSlots];
    __shared__ __align__(16) PhaseDesc d;
    __shared__ float red[2 * kStreamWarps * kRM];
    __shared__ float sred[32], sv[32];
    __shared__ int si[32], last, flag, s_abort, s_pos;
    if (threadIdx.x == 0) {
        for (int s = 0; s < sp.nslots; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kStreamWarps);
        }
        mbar_init_fence();
        s_abort = 0;
        // the position is fixed for the whole step (the argmax phase advances it, after every CTA
        // has passed this point)
        s_pos = sp.state->pos;
    }
    __syncthreads();
    const int pos = s_pos;
    const int warp = threadIdx.x >> 5;
    if (warp == kStreamWarps) {
        if ((threadIdx.x & 31) == 0) stream_producer<HD, GP>(sp, ring, full, empty, pos, &s_abort);
        __syncwarp();
    } else {
        StreamCons cs;
        cs.ring = ring;
        cs.aux = aux;
        cs.full = full;
        cs.empty = empty;
        cs.abort = &s_abort;
        cs.err = &sp.state->err;
        cs.NS = sp.nslots;
        cs.u = 0;
        cs.spin = sp.spin;
        cs.red = red;
        cs.sred = sred;
        cs.buf = 0;
        stream_consumers<HD, GP>(sp, cs, d, pos, sv, si, &last, &flag);
    }
    __syncthreads();   // the producer has drained its copies; the CTA may leave
}

}  // namespace syn
