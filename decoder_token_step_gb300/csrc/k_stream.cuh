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
//                  into a ring of 36 KB shared-memory slots, each completing on an mbarrier; it
//                  waits only for a slot to be released and, before each copy, for the copy D
//                  uses back to have landed. The ring lets it run ahead of the consumers across
//                  phase boundaries; the bound D on copies in flight (2 by default: enough to
//                  cover DRAM latency at the SM's share of HBM bandwidth) keeps the memory queues
//                  short, so the loads the consumers make (x, residuals, the arrival counter) are
//                  not stuck behind many megabytes of queued copies from all SMs.
//   12 consumer    run the phases in order. Before a phase they wait until every CTA has finished
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
constexpr int kMaxTileSlots = 4;                              // slots per GEMV tile (half of kMaxSlots)
constexpr int kStreamThreads = kStreamBlockThreads;           // + the producer and the publisher warp
constexpr int kMaxSlots = 8;
constexpr int kPreRows = 256;                                // GEMV rows per CTA whose bias / residual are prefetched
static_assert(kPreRows <= kConsumerThreads, "one prefetched row per consumer thread");
constexpr unsigned long long kWaitNs = 1000000000ull;         // a ring wait gives up after 1 s
constexpr unsigned long long kGridWaitNs = 2000000000ull;     // the wait for the previous phase, 2 s
constexpr int kNapNs = 64;                                    // pause between polls of the producer and publisher

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
// shared-memory loads by shared-window address (volatile: they stay after the mbarrier waits)
SYN_DEV uint4 lds128_s(uint32_t a) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(a));
    return r;
}
SYN_DEV float4 lds128f_s(uint32_t a) {
    float4 r;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "r"(a));
    return r;
}
SYN_DEV uint16_t lds16_s(uint32_t a) {
    unsigned short r;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(r) : "r"(a));
    return r;
}

SYN_DEV unsigned lds_acquire_u32(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(saddr(p)) : "memory");
    return v;
}
SYN_DEV void sts_release_u32(unsigned *p, unsigned v) {
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(saddr(p)), "r"(v) : "memory");
}

// Bounded wait until done() holds: `spin` < 0 bounds it by wall-clock time (`ns`), else by that many
// polls (0: give up at once; test support). Returns false when it gave up or when `abort` (if
// given) was raised meanwhile. NAP > 0: sleep that many nanoseconds between polls (the producer and
// the publisher, whose polls would otherwise take issue slots and shared-memory bandwidth from the
// consumer warps of their SM sub-partition).
template <int NAP = 0, class Done>
SYN_DEV bool stream_until(Done &&done, int spin, volatile int *abort, unsigned long long ns) {
    if (spin != 0 && done()) return true;   // the usual case: no clock read
    if (spin >= 0) {
        for (int i = 0; i < spin; ++i)
            if (done()) return true;
        return false;
    }
    const unsigned long long deadline = stream_ns() + ns;
    for (unsigned i = 1;; ++i) {
        if (done()) return true;
        if constexpr (NAP > 0) __nanosleep(NAP);
        if ((i & 31u) == 0) {
            if (abort && *abort) return false;
            if (stream_ns() > deadline) return false;
        }
    }
}

// Ring signals in shared memory. Only the publisher warp waits on the copies' mbarriers; the
// consumers and the producer see progress through counters read with acquire loads (an mbarrier
// poll in every consumer warp costs several hundred cycles a slot, in series with its work).
struct StreamSig {
    unsigned ready;                  // uses whose copies have landed (publisher)
    unsigned issued;                 // uses whose copies were issued (producer)
    unsigned prod_done;              // the producer has issued its last copy or stopped
    unsigned done[kStreamWarps];     // uses each consumer warp has finished reading
};

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
SYN_DEV void stream_producer(const StreamParams &sp, uint8_t *ring, uint64_t *full, StreamSig *sig, int pos,
                             volatile int *abort) {
    const int cta = blockIdx.x, ncta = gridDim.x, NS = sp.nslots;
    int *err = &sp.state->err;
    int u = 0;   // slot uses issued
    // the slot of use u once its previous use was released; nullptr when the wait gave up or the
    // consumers aborted
    const int D = sp.inflight;
    auto claim = [&](uint64_t *&bar) -> uint8_t * {
        const int s = u % NS;
        bool got = true;
        if (u >= NS) {   // every consumer warp is done with use u - NS, the slot's previous use
            const unsigned need = (unsigned)(u - NS + 1);
            got = stream_until<kNapNs>([&] {
                unsigned m = 0xffffffffu;
#pragma unroll
                for (int w = 0; w < kStreamWarps; ++w) m = min(m, lds_acquire_u32(&sig->done[w]));
                return m >= need;
            }, sp.spin, abort, kWaitNs);
            // the consumers' generic-proxy reads of the slot are ordered before the copy's writes
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        // at most D copies outstanding: use u - D has landed
        if (got && D < NS && u >= D) got = stream_until<kNapNs>([&] { return lds_acquire_u32(&sig->ready) >= (unsigned)(u - D + 1); }, sp.spin, abort, kWaitNs);
        if (!got) {
            if (!*abort) atomicOr(err, ERR_STREAM);
            *abort = 1;
            return nullptr;
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
                        if (g.gstride == (int)rb) {   // whole rows: one copy of codes, one of scales
                            bulk_g2s(dst, static_cast<const uint8_t *>(W.codes) + (size_t)r * rb, cb, bar);
                            if (q) bulk_g2s(dst + (size_t)g.rs * rb, W.scales + (size_t)r * ss, sb, bar);
                        } else {                      // a column slice: each row's part on its own
                            for (int j = 0; j < cnt; ++j) {
                                bulk_g2s(dst + (size_t)j * rb, static_cast<const uint8_t *>(W.codes) + (size_t)(r + j) * g.gstride, (unsigned)rb, bar);
                                if (q)
                                    bulk_g2s(dst + (size_t)g.rs * rb + (size_t)j * ss * 2, W.scales + (size_t)(r + j) * g.sstride,
                                             (unsigned)(ss * 2), bar);
                            }
                        }
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
                    sts_release_u32(&sig->issued, (unsigned)u);
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
                        sts_release_u32(&sig->issued, (unsigned)u);
                    }
                }
            }
        }
    }
    // the publisher waits for every issued copy before the CTA leaves
    sts_release_u32(&sig->prod_done, 1u);
}

// The publisher: waits for the ring's copies in issue order and publishes their count in `ready`.
// It runs until the producer has stopped and every issued copy has landed (each wait bounded by
// wall-clock time whatever the abort state: no copy may land after the CTA has left).
SYN_DEV void stream_publisher(const StreamParams &sp, uint64_t *full, StreamSig *sig, volatile int *abort) {
    const int NS = sp.nslots;
    int *err = &sp.state->err;
    unsigned v = 0;
    unsigned long long idle_since = 0;
    for (unsigned i = 0;; ++i) {
        const unsigned iss = lds_acquire_u32(&sig->issued);
        if (v < iss) {
            const int s = (int)(v % (unsigned)NS);
            const unsigned par = (v / (unsigned)NS) & 1u;
            if (!stream_until<kNapNs>([&] { return mbar_try(&full[s], par); }, -1, nullptr, kWaitNs)) {
                atomicOr(err, ERR_STREAM);
                *abort = 1;
            }
            sts_release_u32(&sig->ready, ++v);
            idle_since = 0;
            continue;
        }
        if (lds_acquire_u32(&sig->prod_done) && v >= lds_acquire_u32(&sig->issued)) break;
        __nanosleep(kNapNs);
        if ((i & 63u) == 0) {   // the producer's own waits are bounded: it always ends
            const unsigned long long t = stream_ns();
            if (!idle_since) idle_since = t;
            else if (t - idle_since > 4 * kGridWaitNs) {
                atomicOr(err, ERR_STREAM);
                *abort = 1;
                break;
            }
        }
    }
}

// ------------------------------------------------------------------------------- consumers
struct StreamCons {
    uint8_t *ring;
    float *aux;
    StreamSig *sig;
    volatile int *abort;
    int *err;
    int NS;
    int u;          // slot uses consumed
    int us;         // u % NS
    int spin;       // wait bound (see stream_until)
    float *red;     // [kRedBufs][kStreamWarps][8] tile partial sums
    int *tile_cnt;  // [kRedBufs] warps done with the tile that uses the buffer
    float *pre;     // [2 * kPreRows] bias / residual of the CTA's rows of a GEMV phase
    float *sred;    // 32 floats
    int buf;
    unsigned long long *trace;   // this phase's 5 trace stamps (CTA 0 when profiling), else nullptr
    // ring slot of use u + k (k < kMaxTileSlots <= NS)
    SYN_DEV int slot_of(int k) const {
        const int s = us + k;
        return s >= NS ? s - NS : s;
    }
    // wait until uses u .. u + n - 1 have landed (whole warp; false once aborted): lane 0 polls the
    // ready count, then the warp barrier orders every lane's shared-memory reads after its acquire
    SYN_DEV bool wait_tile(int n) {
        bool ok = true;
        if ((threadIdx.x & 31) == 0) {
            const unsigned need = (unsigned)(u + n);
            ok = !*abort && stream_until([&] { return lds_acquire_u32(&sig->ready) >= need; }, spin, abort, kWaitNs);
            if (!ok) {
                if (!*abort) atomicOr(err, ERR_STREAM);
                *abort = 1;
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
        __syncwarp();
        return ok;
    }
    SYN_DEV uint8_t *slot(int k) const { return ring + (size_t)slot_of(k) * kSlotBytes; }
    // this warp is done reading uses u .. u + n - 1
    SYN_DEV void release(int n) {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) sts_release_u32(&sig->done[threadIdx.x >> 5], (unsigned)(u + n));
        u += n;
        us = slot_of(n);
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
// E16: weights per 16 bytes of a row; scales per 32 weights (GGUF blocks)
template <> struct ChunkShape<W_Q8_0> { static constexpr int E16 = 16, SPC = 1; };
template <> struct ChunkShape<W_Q4_0> { static constexpr int E16 = 32, SPC = 2; };
template <> struct ChunkShape<W_F16> { static constexpr int E16 = 8, SPC = 0; };
template <> struct ChunkShape<W_F32> { static constexpr int E16 = 4, SPC = 0; };

template <int WT> SYN_DEV float dot16(const uint4 c, const float *x) {
    if constexpr (WT == W_Q8_0) return dot16_q8(c, x);
    else if constexpr (WT == W_Q4_0) return dot16_q4(c, x);
    else if constexpr (WT == W_F16) return dot16_f16(c, x);
    else return dot16_f32(c, x);
}

constexpr int kRedBufs = 12;   // tile reduction buffers (more than ring slots: no warp laps another)

// The tiles of one GEMV phase on the consumer threads (x already staged). A consumer thread owns
// chunks of NH x 16 bytes of the rows (chunk c, c + stride, ...) and computes RPT rows of the
// tile (rows grp, grp + P, ...): the rows are unrolled with no branch between them (absent rows
// read a valid slot row and are masked), so that their independent FMA chains interleave; the
// chunk's x values are loaded once per tile and serve all RPT rows. With NH = 2 a lane reads the
// two 16-byte halves of its chunk in a lane-dependent order, which keeps the shared loads free of
// bank conflicts. Partial sums: a warp reduce-scatter, one row of partials per warp in shared
// memory, and the last warp to finish a tile sums them in warp order (deterministic) and writes
// the outputs; no block-wide barrier per tile.
template <int WT, int RPT, int NH>
SYN_DEV void stream_gemv_tiles(const PhaseDesc &d, StreamCons &cs, int cta, int ncta, const float (&xa)[ChunkShape<WT>::E16],
                               const float (&xb)[ChunkShape<WT>::E16], float inv, const float *pre, int pre_v0, int pre_n) {
    constexpr int E16 = ChunkShape<WT>::E16, SPC = ChunkShape<WT>::SPC;
    constexpr int RS = RPT == 6 ? 8 : RPT == 3 ? 4 : RPT;   // reduce-scatter width (a power of two)
    const GemvParams &p = d.gemv;
    const StreamGemv &g = d.sg;
    const bool gu = p.gate_up != 0;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rb = (int)p.seg[0].W.row_bytes;
    const int ss = (int)p.seg[0].W.scale_stride;
    const int C = g.C, rs = g.rs, P = g.P, hrows = rs / 2, wg = g.wg;
    const int cap = g.slots * rs;                        // positions of a full tile
    const int grp = P > 1 ? warp / wg : 0;
    const int c = P > 1 ? (warp - grp * wg) * 32 + lane : tid;   // this thread's chunk
    const bool active = grp < P && c < C;
    const int h0 = NH == 2 ? (lane >> 2) & 1 : 0;       // which half of the chunk this lane reads first
    const uint32_t ring_s = saddr(cs.ring);
    const int cbyte = c * 16 * NH;                       // the chunk's first byte in a row
    const int cscale = SPC == 1 ? ((c * NH) >> 1) * 2 : (c * NH) * 2;   // its first scale (bytes)
    // A tile position t = k * rs + j is row j of slot k; its list index inside the tile (the row,
    // or for gate/up the pair) is t, or k * hrows + j mod hrows.
    auto list_of = [&](int k, int j) { return gu ? k * hrows + (j < hrows ? j : j - hrows) : k * rs + j; };
    // this thread's rows (positions grp + P * i), fixed for the phase and packed two registers a
    // row: ro = byte offset of the chunk's codes inside the slot | offset of its scales << 16 (both
    // below kSlotBytes < 2^16); rl = slot index (2 bits) | list index << 2 (127: never a row)
    static_assert(kSlotBytes < 65536 && kMaxTileSlots <= 4, "packed row offsets");
    uint32_t ro[RPT], rl[RPT];
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
        const int t = grp + P * i;
        const int k = t / rs, j = t - k * rs;
        const bool v = active && t < cap;
        const uint32_t off = (uint32_t)((v ? j * rb : 0) + cbyte + h0 * 16);
        const uint32_t soff = (uint32_t)(rs * rb + (v ? j * ss * 2 : 0) + cscale);
        ro[i] = off | soff << 16;
        rl[i] = v ? (uint32_t)k | (uint32_t)list_of(k, j) << 2 : 127u << 2;
    }
    // this lane's output positions for the tile epilogue (t = lane, lane + 32; cap <= 64): list
    // index (-1: none), and packed bytes: row group of its sums, index of the partial in each warp,
    // the same for the up half of a gate/up pair
    int el[2];
    uint32_t ep[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int t = lane + 32 * e;
        const int k = t / rs, j = t - k * rs;
        const bool v = t < cap && (!gu || j < hrows);
        el[e] = v ? list_of(k, j) : -1;
        ep[e] = (uint32_t)(t % P) | (uint32_t)(t / P) << 8 | (uint32_t)((t + hrows) % P) << 16 | (uint32_t)((t + hrows) / P) << 24;
    }

    GemvTiles T(g, gu, cta, ncta);
    int seg, row0, n;
    while (true) {
        const int vstart = T.v;   // list position of the tile's first row
        if (!T.next(g, seg, row0, n)) break;
        const int nsl = gemv_tile_slots(g, gu, n);
        const bool okw = cs.wait_tile(nsl);
        float acc[RS];
#pragma unroll
        for (int i = 0; i < RS; ++i) acc[i] = 0.f;
        unsigned vmask = 0;
#pragma unroll
        for (int i = 0; i < RPT; ++i) vmask |= (unsigned)((int)(rl[i] >> 2) < n) << i;
        if (okw && vmask) {
            // byte addresses of this thread's rows (absent rows read the first slot; masked below)
            uint32_t ad[RPT], sd[RPT];
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const uint32_t base = ring_s + (uint32_t)(cs.slot_of((vmask >> i) & 1u ? (int)(rl[i] & 3u) : 0) * kSlotBytes);
                ad[i] = base + (ro[i] & 0xffffu);
                sd[i] = base + (ro[i] >> 16);
            }
            float dsc[RPT];
            if constexpr (SPC == 1) {   // one scale per 32 bytes of codes
#pragma unroll
                for (int i = 0; i < RPT; ++i) dsc[i] = half_bits_to_float(lds16_s(sd[i]));
            }
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) {
                const float *x = hh ? xb : xa;
                const int dh = NH == 2 ? (hh ? (1 - 2 * h0) * 16 : 0) : 0;   // the other half
#pragma unroll
                for (int i = 0; i < RPT; ++i) {
                    const uint4 cw = lds128_s(ad[i] + dh);
                    const float dv = dot16<WT>(cw, x);
                    if constexpr (SPC == 0) {
                        acc[i] += dv;
                    } else if constexpr (SPC == 1) {
                        acc[i] = fmaf(dsc[i], dv, acc[i]);
                    } else {   // one scale per 16 bytes of codes (a Q4_0 block)
                        acc[i] = fmaf(half_bits_to_float(lds16_s(sd[i] + (NH == 2 ? (hh ? 1 - h0 : h0) * 2 : 0))), dv, acc[i]);
                    }
                }
            }
        }
        cs.release(nsl);
#pragma unroll
        for (int i = 0; i < RPT; ++i) acc[i] = (vmask >> i) & 1u ? acc[i] : 0.f;
        // ---- this warp's partial sums, then the last warp of the tile sums the warps in order
        const float v = reduce_scatter<RS>(acc, lane);
        const int b = cs.buf;
        float *red = cs.red + b * kStreamWarps * 8;
        constexpr int LPV = 32 / RS;                      // lanes holding the same value
        if ((lane & (LPV - 1)) == 0) red[warp * 8 + lane / LPV] = v;
        __syncwarp();
        int last = 0;
        if (lane == 31) {   // a lane without epilogue stores of its own (tiles have fewer than 32 rows)
            __threadfence_block();
            last = atomicAdd(&cs.tile_cnt[b], 1) == kStreamWarps - 1;
        }
        last = __shfl_sync(0xffffffffu, last, 31);
        if (last) {
            __threadfence_block();
            const GemvSeg &S = p.seg[gu ? 0 : seg];
            float *out = S.out;
            const bool use_pre = pre != nullptr;
            const float *bias = S.bias, *bias_u = gu ? p.seg[1].bias : nullptr;
            const bool add = S.epi == EPI_ADD;
            const int act = p.act;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int lt = el[e];
                if (lt < 0 || lt >= n) continue;
                float sum = 0.f, usum = 0.f;
                const uint32_t q = ep[e];
                const float *rs0 = red + (int)(q & 0xffu) * wg * 8 + (int)((q >> 8) & 0xffu);
#pragma unroll
                for (int w2 = 0; w2 < kStreamWarps; ++w2)
                    if (w2 < wg) sum += rs0[w2 * 8];
                if (gu) {
                    const float *rs1 = red + (int)((q >> 16) & 0xffu) * wg * 8 + (int)(q >> 24);
#pragma unroll
                    for (int w2 = 0; w2 < kStreamWarps; ++w2)
                        if (w2 < wg) usum += rs1[w2 * 8];
                }
                const int r = row0 + lt;                       // row (pair) inside its segment
                const int lv = vstart + lt - pre_v0;           // position in the CTA's list range
                const bool pv = use_pre && lv >= 0 && lv < pre_n;
                if (gu) {
                    const float bg = pv ? pre[lv] : (bias ? bias[r] : 0.f);
                    const float bu = pv ? pre[pre_n + lv] : (bias_u ? bias_u[r] : 0.f);
                    out[r] = apply_act(act, sum * inv + bg) * (usum * inv + bu);
                } else {
                    float y = sum * inv;
                    if (pv) {
                        y += pre[lv] + pre[pre_n + lv];          // bias, residual
                    } else {
                        if (bias) y += bias[r];
                        if (add) y += __ldcg(out + r);
                    }
                    out[r] = y;
                }
            }
            __syncwarp();
            if (lane == 31) cs.tile_cnt[b] = 0;
        }
        cs.buf = (b + 1) % kRedBufs;
    }
}

// One GEMV phase on the consumer threads. Each consumer thread owns one chunk (16 or 32 bytes) of
// every row for the whole phase: it loads that chunk's x values (times the norm weight) into
// registers once, the halves in the order its lane reads the codes; the sum of squares for the
// rms norm comes from the threads of the first row group, which together hold each chunk once.
// The bias and residual of the CTA's rows go to shared memory. Then the tiles.
template <int WT, int NH>
SYN_DEV void stream_gemv_nh(const PhaseDesc &d, StreamCons &cs, int cta, int ncta) {
    constexpr int E16 = ChunkShape<WT>::E16, ECH = E16 * NH;
    const GemvParams &p = d.gemv;
    const StreamGemv &g = d.sg;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int K = (int)p.seg[0].W.K;
    const int P = g.P;
    const int grp = P > 1 ? warp / g.wg : 0;
    const int c = P > 1 ? (warp - grp * g.wg) * 32 + lane : tid;
    const bool has = grp < P && c < g.C;
    const int h0 = NH == 2 ? (lane >> 2) & 1 : 0;
    // bias and residual of this CTA's rows (list positions v0 .. v1-1), loads issued first:
    // pre[0 .. n) bias (gate bias for gate/up), pre[n .. 2n) residual (up bias for gate/up)
    const bool gu = p.gate_up != 0;
    const int v0 = (int)((int64_t)g.rows * cta / ncta), v1 = (int)((int64_t)g.rows * (cta + 1) / ncta);
    const int npre = v1 - v0;
    bool need = false;
    for (int i = 0; i < p.nseg; ++i) need = need || p.seg[i].bias || p.seg[i].epi == EPI_ADD;
    float *pre = (need && npre <= kPreRows) ? cs.pre : nullptr;   // kPreRows <= kConsumerThreads: one entry per thread
    float pre_a = 0.f, pre_b = 0.f;
    if (pre && tid < npre) {
        const int v = v0 + tid;
        if (gu) {
            pre_a = p.seg[0].bias ? p.seg[0].bias[v] : 0.f;
            pre_b = p.seg[1].bias ? p.seg[1].bias[v] : 0.f;
        } else {
            const int sg = (v >= g.seg_end[0]) + (v >= g.seg_end[1]);
            const int r = v - (sg == 0 ? 0 : g.seg_end[sg - 1]);
            const GemvSeg &S = p.seg[sg];
            pre_a = S.bias ? S.bias[r] : 0.f;
            pre_b = S.epi == EPI_ADD ? __ldcg(S.out + r) : 0.f;
        }
    }
    // this thread's chunk of x: elements c * ECH + half * E16 + e (zero past K)
    float xa[E16], xb[E16];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        float *xv = hh ? xb : xa;
        const int half = NH == 2 ? (hh ? 1 - h0 : h0) : 0;
        const int e0 = c * ECH + half * E16;
#pragma unroll
        for (int j = 0; j < E16 / 4; ++j) {
            const int i = e0 + 4 * j;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (has && (NH == 2 || hh == 0) && i < K) v = __ldcg(reinterpret_cast<const float4 *>(p.x + i));
            xv[4 * j] = v.x; xv[4 * j + 1] = v.y; xv[4 * j + 2] = v.z; xv[4 * j + 3] = v.w;
        }
    }
    float sq = 0.f;
    if (grp == 0 && has) {
#pragma unroll
        for (int e = 0; e < E16; ++e) sq = fmaf(xa[e], xa[e], fmaf(xb[e], xb[e], sq));
    }
    if (p.norm_w && has) {
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
            float *xv = hh ? xb : xa;
            const int e0 = c * ECH + (NH == 2 ? (hh ? 1 - h0 : h0) : 0) * E16;
#pragma unroll
            for (int j = 0; j < E16 / 4; ++j) {
                const int i = e0 + 4 * j;
                if (i < K) {
                    const float4 w = *reinterpret_cast<const float4 *>(p.norm_w + i);
                    xv[4 * j] *= w.x; xv[4 * j + 1] *= w.y; xv[4 * j + 2] *= w.z; xv[4 * j + 3] *= w.w;
                }
            }
        }
    }
    if (pre && tid < npre) {
        pre[tid] = pre_a;
        pre[npre + tid] = pre_b;
    }
    // the block sum's barriers also publish pre to every consumer
    sq = block_sum<ConsumerThreads>(sq, cs.sred);
    const float inv = p.norm_w ? 1.f / sqrtf(sq / (float)K + p.eps) : 1.f;
    if (cs.trace && threadIdx.x == 0) cs.trace[3] = stream_ns();
    switch (g.rpt) {
    case 2: stream_gemv_tiles<WT, 2, NH>(d, cs, cta, ncta, xa, xb, inv, pre, v0, npre); break;
    case 3: stream_gemv_tiles<WT, 3, NH>(d, cs, cta, ncta, xa, xb, inv, pre, v0, npre); break;
    case 4: stream_gemv_tiles<WT, 4, NH>(d, cs, cta, ncta, xa, xb, inv, pre, v0, npre); break;
    case 6: stream_gemv_tiles<WT, 6, NH>(d, cs, cta, ncta, xa, xb, inv, pre, v0, npre); break;
    default: stream_gemv_tiles<WT, 8, NH>(d, cs, cta, ncta, xa, xb, inv, pre, v0, npre); break;
    }
    if (cs.trace && threadIdx.x == 0) cs.trace[4] = stream_ns();
}

// The phase functions are not inlined: each gets its own register allocation, so that the
// registers one phase kind needs (a GEMV's x chunk and row state, the attention's query heads and
// accumulators) do not crowd another's. The ring state travels by value.
template <int WT> __device__ __noinline__ StreamCons stream_gemv(const PhaseDesc &d, StreamCons cs, int cta, int ncta) {
    if (d.sg.cb == 16) stream_gemv_nh<WT, 1>(d, cs, cta, ncta);
    else stream_gemv_nh<WT, 2>(d, cs, cta, ncta);
    return cs;
}

// barrier over the kAttnWarps warps that run the attention (named barrier 2)
SYN_DEV void attn_group_sync() { asm volatile("bar.sync 2, %0;" ::"r"(kAttnThreads) : "memory"); }

// One attention phase on the consumer threads (decode: one query row at position pos). Warps
// 0 .. kAttnWarps-1 compute (the shapes of attn_dev.cuh); the other consumer warps walk the same
// ring tiles and release them.
template <int HD, int GP, class KV>
__device__ __noinline__ StreamCons stream_attn(const PhaseDesc &d, StreamCons cs, int cta, int ncta, int pos) {
    using Sh = AttnShape<HD, GP>;
    constexpr int EL = Sh::EL, KB = Sh::KB, TK = kAttnWarps * KB;
    const AttnParams &a = d.attn;
    const HeadsParams &h = a.heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool worker = warp < kAttnWarps;
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
        if (!worker) {
            for (int t0 = start; t0 < old_end; t0 += TK) {
                cs.wait_tile(2);
                cs.release(2);
            }
            continue;
        }
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
            float kr[KB][EL], vr[EL];
#pragma unroll
            for (int j = 0; j < KB; ++j)
#pragma unroll
                for (int e = 0; e < EL; ++e) kr[j][e] = 0.f;
            KV *kd = static_cast<KV *>(const_cast<void *>(a.kcache)) + ((size_t)g * a.max_ctx + pos) * HD + lane * EL;
            KV *vd = static_cast<KV *>(const_cast<void *>(a.vcache)) + ((size_t)g * a.max_ctx + pos) * HD + lane * EL;
            if (a.fuse_heads) {
#pragma unroll
                for (int e = 0; e < EL; ++e) {
                    kr[0][e] = __ldcg(h.k + (size_t)g * HD + lane * EL + e);
                    vr[e] = __ldcg(h.v + (size_t)g * HD + lane * EL + e);
                    if (h.bv) vr[e] += h.bv[(size_t)g * HD + lane * EL + e];
                }
                head_transform<HD>(kr[0], h.bk ? h.bk + (size_t)g * HD : nullptr, h.wk, h.rope_k, rcs, h.rope_adjacent, h.eps);
#pragma unroll
                for (int e = 0; e < EL; ++e) {
                    st_kv(kd + e, kr[0][e]);
                    st_kv(vd + e, vr[e]);
                }
                // the cache holds the rounded values (f16 cache): attend to what was stored
                if constexpr (sizeof(KV) == 2) {
#pragma unroll
                    for (int e = 0; e < EL; ++e) {
                        kr[0][e] = __half2float(__float2half_rn(kr[0][e]));
                        vr[e] = __half2float(__float2half_rn(vr[e]));
                    }
                }
            } else {
#pragma unroll
                for (int e = 0; e < EL; ++e) {
                    if constexpr (sizeof(KV) == 2) {
                        kr[0][e] = __half2float(__ushort_as_half(__ldcg(reinterpret_cast<const unsigned short *>(kd + e))));
                        vr[e] = __half2float(__ushort_as_half(__ldcg(reinterpret_cast<const unsigned short *>(vd + e))));
                    } else {
                        kr[0][e] = __ldcg(reinterpret_cast<const float *>(kd + e));
                        vr[e] = __ldcg(reinterpret_cast<const float *>(vd + e));
                    }
                }
            }
            attn_step_v<HD, GP>(q, kr, [&](int j, float (&v)[EL]) {
#pragma unroll
                for (int e = 0; e < EL; ++e) v[e] = j == 0 ? vr[e] : 0.f;
            }, 1, G, scale, m_run, l_run, o);
        }
        for (int t0 = start; t0 < old_end; t0 += TK) {
            const bool okw = cs.wait_tile(2);
            const int tw = t0 + warp * KB;
            const int nk = min(KB, old_end - tw);
            if (okw && nk > 0) {
                const KV *sk = reinterpret_cast<const KV *>(cs.slot(0)) + warp * KB * HD + lane * EL;
                const KV *sv = reinterpret_cast<const KV *>(cs.slot(1)) + warp * KB * HD + lane * EL;
                float kr[KB][EL];
#pragma unroll
                for (int j = 0; j < KB; ++j) {
                    if (j < nk) {
                        lds_row<EL>(kr[j], sk + j * HD);
                    } else {
#pragma unroll
                        for (int e = 0; e < EL; ++e) kr[j][e] = 0.f;
                    }
                }
                // value rows past nk hold another tile's data (or none): read as zeros
                attn_step_v<HD, GP>(q, kr, [&](int j, float (&v)[EL]) {
                    if (j < nk) {
                        lds_row<EL>(v, sv + j * HD);
                    } else {
#pragma unroll
                        for (int e = 0; e < EL; ++e) v[e] = 0.f;
                    }
                }, nk, G, scale, m_run, l_run, o);
            }
            cs.release(2);
        }
        // merge the warps and the slices (the aux region is the merge scratch)
        attn_group_sync();
        attn_finish<HD, GP>(a, S, g, split, 0, cs.aux, m_run, l_run, o, [] { attn_group_sync(); });
    }
    return cs;
}

// a further column slice of a matmul depends only on this CTA's previous phase
SYN_DEV bool d_no_wait(const StreamParams &sp, int ph) { return __ldg(&sp.phases[ph].no_wait) != 0; }

template <int HD, int GP>
SYN_DEV void stream_consumers(const StreamParams &sp, StreamCons &cs, PhaseDesc &d, int pos, float *sv, int *si,
                              int *last, int *flag) {
    const int cta = blockIdx.x, ncta = gridDim.x;
    const bool tr = sp.trace && cta == 0 && threadIdx.x == 0;
    for (int ph = 0; ph < sp.nphases; ++ph) {
        cs.trace = sp.trace && cta == 0 ? sp.trace + 5 * ph : nullptr;
        // the phase descriptor into shared memory (every consumer is past the previous phase)
        {
            const int4 *src = reinterpret_cast<const int4 *>(sp.phases + ph);
            int4 *dst = reinterpret_cast<int4 *>(&d);
            for (int i = threadIdx.x; i < (int)(sizeof(PhaseDesc) / 16); i += kConsumerThreads) dst[i] = __ldg(src + i);
        }
        if (tr) sp.trace[5 * ph] = stream_ns();
        if (threadIdx.x == 0) {
            // every CTA has finished phases 0 .. ph-1 (bounded; gives up early once any CTA failed)
            if (ph > 0 && !*cs.abort && !d_no_wait(sp, ph)) {
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
        if (tr) sp.trace[5 * ph + 1] = sp.trace[5 * ph + 3] = sp.trace[5 * ph + 4] = stream_ns();
        const bool run = !*flag;
        switch (d.kind) {
        case PH_GEMV:
            // even when aborted, the tiles are walked (without waiting) to keep the ring accounting
            switch (d.gemv.seg[0].W.wtype) {
            case W_Q8_0: cs = stream_gemv<W_Q8_0>(d, cs, cta, ncta); break;
            case W_Q4_0: cs = stream_gemv<W_Q4_0>(d, cs, cta, ncta); break;
            case W_F16: cs = stream_gemv<W_F16>(d, cs, cta, ncta); break;
            default: cs = stream_gemv<W_F32>(d, cs, cta, ncta); break;
            }
            break;
        case PH_ATTN:
            if (d.attn.kv_f16) cs = stream_attn<HD, GP, __half>(d, cs, cta, ncta, pos);
            else cs = stream_attn<HD, GP, float>(d, cs, cta, ncta, pos);
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
        if (tr) sp.trace[5 * ph + 2] = stream_ns();
    }
}

// HD, GP: head dimension and padded query-group size of the attention phases (one model has one
// of each); every weight type is handled inside.
template <int HD, int GP>
__global__ void __launch_bounds__(kStreamThreads, 1) k_stream(const StreamParams sp) {
    extern __shared__ uint8_t stream_smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(stream_smem_raw) + 127) & ~uintptr_t(127));
    float *aux = reinterpret_cast<float *>(ring + (size_t)sp.nslots * kSlotBytes);
    __shared__ __align__(8) uint64_t full[kMaxSlots];
    __shared__ StreamSig sig;
    __shared__ __align__(16) PhaseDesc d;
    __shared__ float red[kRedBufs * kStreamWarps * 8];
    __shared__ float pre[2 * kPreRows];
    __shared__ float sred[32], sv[32];
    __shared__ int si[32], tile_cnt[kRedBufs], last, flag, s_abort, s_pos;
    if (threadIdx.x == 0) {
        for (int s = 0; s < sp.nslots; ++s) mbar_init(&full[s], 1);
        mbar_init_fence();
        sig.ready = sig.issued = sig.prod_done = 0;
        for (int w = 0; w < kStreamWarps; ++w) sig.done[w] = 0;
        for (int i = 0; i < kRedBufs; ++i) tile_cnt[i] = 0;
        s_abort = 0;
        // the position is fixed for the whole step (the argmax phase advances it, after every CTA
        // has passed this point)
        s_pos = sp.state->pos;
    }
    __syncthreads();
    const int pos = s_pos;
    const int warp = threadIdx.x >> 5;
    if (warp == kStreamWarps) {
        if ((threadIdx.x & 31) == 0) stream_producer<HD, GP>(sp, ring, full, &sig, pos, &s_abort);
        __syncwarp();
    } else if (warp == kStreamWarps + 1) {
        if ((threadIdx.x & 31) == 0) stream_publisher(sp, full, &sig, &s_abort);
        __syncwarp();
    } else {
        StreamCons cs;
        cs.ring = ring;
        cs.aux = aux;
        cs.sig = &sig;
        cs.abort = &s_abort;
        cs.err = &sp.state->err;
        cs.NS = sp.nslots;
        cs.u = 0;
        cs.us = 0;
        cs.spin = sp.spin;
        cs.red = red;
        cs.tile_cnt = tile_cnt;
        cs.pre = pre;
        cs.sred = sred;
        cs.buf = 0;
        cs.trace = nullptr;
        stream_consumers<HD, GP>(sp, cs, d, pos, sv, si, &last, &flag);
    }
    __syncthreads();   // the producer has drained its copies; the CTA may leave
}

}  // namespace syn
