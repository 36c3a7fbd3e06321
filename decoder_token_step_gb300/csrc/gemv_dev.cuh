// gemv_dev.cuh -- the weight-streaming GEMV of the decode step as a device function (the kernel is
// in k_gemv.cu).
//
// `matmul(h, W)` of "Local inference and architectures" (synsema.dev, section "The format"), with
// weights "multiplied in f32" (section "Choosing the engine"): every weight is decoded to its exact
// f32 value in registers and multiplied with the f32 activation; partial sums are f32.
//
// At batch size 1 the product is bound by reading W from HBM once, so the code is built around the
// load stream and keeps the arithmetic per weight small enough to stay under it:
//   * each warp owns 2 rows at a time (the two rows of a fused gate/up pair, or 2 consecutive
//     rows); lane l reads the 32-byte chunks l, l+32, ... of both rows with 256-bit loads (one
//     whole Q8_0 block per load), and the next batch of loads is issued before the current one is
//     consumed (register double buffering);
//   * the input vector is staged once per CTA in shared memory, lane-interleaved so that every
//     float4 read is bank-conflict free, and both rows share each x read;
//   * codes become floats without conversion instructions (a byte in the mantissa of 2^23, then
//     one packed f32x2 subtraction), and products accumulate with packed f32x2 FMAs;
//   * an optional RMSNorm of the input is folded in: x * w is staged and the dot product is scaled
//     by 1/rms at the end (fused `rms_norm` step); the epilogue adds a bias, stores or accumulates
//     into the destination (fused `add_bias` and residual `add`), or forms act(gate) * up;
//   * each CTA takes a contiguous, balanced range of row pairs, and its first weight loads are
//     issued before it waits for the previous kernel.
#pragma once

#include "device_common.cuh"

namespace syn {


struct U8 { uint32_t w[8]; };

SYN_DEV U8 ld32(const void *p) {
    U8 r;
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]), "=r"(r.w[5]),
                   "=r"(r.w[6]), "=r"(r.w[7])
                 : "l"(p));
    return r;
}

// byte `which` of w placed in the low mantissa of 2^23: the float 2^23 + byte, exactly
SYN_DEV float magic(uint32_t w, int which) { return __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u | (uint32_t)which)); }

// Dot product of one 32-byte chunk of a row with its x values. x slots: float4 number j of lane l
// of a slab sits at xs[j * 128 + l * 4].
template <int WT> struct Chunk32;

// Q8_0: 32 offset-binary codes (q + 128) = one whole block; the block scale is applied by the caller.
template <> struct Chunk32<W_Q8_0> {
    static constexpr int E = 32;
    static SYN_DEV float dot(const U8 &c, const float *xs) {
        float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
        const float2 bias = make_float2(-8388736.f, -8388736.f);  // 2^23 + 128
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 x = *reinterpret_cast<const float4 *>(xs + i * 128);
            const float2 q01 = __fadd2_rn(make_float2(magic(c.w[i], 0), magic(c.w[i], 1)), bias);
            const float2 q23 = __fadd2_rn(make_float2(magic(c.w[i], 2), magic(c.w[i], 3)), bias);
            a0 = __ffma2_rn(q01, make_float2(x.x, x.y), a0);
            a1 = __ffma2_rn(q23, make_float2(x.z, x.w), a1);
        }
        return (a0.x + a0.y) + (a1.x + a1.y);
    }
};

// Q4_0: two whole blocks; word i of block b holds elements 4i..4i+3 in its low nibbles and
// 16+4i..16+4i+3 in its high nibbles; codes decode to code - 8. Returns both block sums.
template <> struct Chunk32<W_Q4_0> {
    static constexpr int E = 64;
    static SYN_DEV float2 dot2(const U8 &c, const float *xs) {
        float s[2];
        const float2 bias = make_float2(-8388616.f, -8388616.f);  // 2^23 + 8
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
            for (int ii = 0; ii < 4; ++ii) {
                const uint32_t w = c.w[b * 4 + ii];
                const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
                const float4 xl = *reinterpret_cast<const float4 *>(xs + (b * 8 + ii) * 128);
                const float4 xh = *reinterpret_cast<const float4 *>(xs + (b * 8 + 4 + ii) * 128);
                a0 = __ffma2_rn(__fadd2_rn(make_float2(magic(lo, 0), magic(lo, 1)), bias), make_float2(xl.x, xl.y), a0);
                a1 = __ffma2_rn(__fadd2_rn(make_float2(magic(lo, 2), magic(lo, 3)), bias), make_float2(xl.z, xl.w), a1);
                a0 = __ffma2_rn(__fadd2_rn(make_float2(magic(hi, 0), magic(hi, 1)), bias), make_float2(xh.x, xh.y), a0);
                a1 = __ffma2_rn(__fadd2_rn(make_float2(magic(hi, 2), magic(hi, 3)), bias), make_float2(xh.z, xh.w), a1);
            }
            s[b] = (a0.x + a0.y) + (a1.x + a1.y);
        }
        return make_float2(s[0], s[1]);
    }
};

template <> struct Chunk32<W_F16> {
    static constexpr int E = 16;
    static SYN_DEV float dot(const U8 &c, const float *xs) {
        float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 x = *reinterpret_cast<const float4 *>(xs + i * 128);
            const float2 w0 = __half22float2(*reinterpret_cast<const __half2 *>(&c.w[2 * i]));
            const float2 w1 = __half22float2(*reinterpret_cast<const __half2 *>(&c.w[2 * i + 1]));
            a0 = __ffma2_rn(w0, make_float2(x.x, x.y), a0);
            a1 = __ffma2_rn(w1, make_float2(x.z, x.w), a1);
        }
        return (a0.x + a0.y) + (a1.x + a1.y);
    }
};

template <> struct Chunk32<W_F32> {
    static constexpr int E = 8;
    static SYN_DEV float dot(const U8 &c, const float *xs) {
        float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float4 x = *reinterpret_cast<const float4 *>(xs + i * 128);
            a0 = __ffma2_rn(make_float2(__uint_as_float(c.w[4 * i]), __uint_as_float(c.w[4 * i + 1])), make_float2(x.x, x.y), a0);
            a1 = __ffma2_rn(make_float2(__uint_as_float(c.w[4 * i + 2]), __uint_as_float(c.w[4 * i + 3])), make_float2(x.z, x.w), a1);
        }
        return (a0.x + a0.y) + (a1.x + a1.y);
    }
};

// shared-memory slot of x element i (32-byte chunks of E elements, lane-interleaved float4s)
template <int E> SYN_DEV int xs_slot(int i) {
    const int g = i / (32 * E), rem = i % (32 * E), l = rem / E, e = rem % E;
    return g * 32 * E + (e >> 2) * 128 + l * 4 + (e & 3);
}

// The GEMV work of one CTA of kWarps warps: row groups [g0, g1) of groups_total, split evenly over
// ncta CTAs. A warp task is a group of kR rows (kR = 2 for the gate/up pairs); a lane reads kU
// 32-byte chunks of each row per batch. `wait()` is called exactly once, after the first weight
// loads are issued and before anything that depends on earlier work (x, the residual) is read or
// any output is written. p.gend must count groups of kR rows (gemv_set_groups(p, kR)).
template <int WT, bool GATE_UP, int kR, int kU, int kWarps, bool PRE, class Wait>
SYN_DEV void gemv_cta(const GemvParams &p, const GemvPre &pre, int groups_total, int cta, int ncta, float *xs, float *red,
                      Wait &&wait) {
    constexpr int kThreads = kWarps * 32;
    constexpr int E = Chunk32<WT>::E;
    constexpr bool Q = (WT == W_Q8_0 || WT == W_Q4_0);
    constexpr int SPC = WT == W_Q4_0 ? 2 : 1;  // block scales per chunk
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int K = (int)p.seg[0].W.K;
    const int chunks = (int)(p.seg[0].W.row_bytes / 32);
    const int slabs = (chunks + 31) / 32;
    const int xs_len = slabs * 32 * E;
    const int nbat = (slabs + kU - 1) / kU;  // batches per row pair
    const int g0 = (int)((int64_t)groups_total * cta / ncta), g1 = (int)((int64_t)groups_total * (cta + 1) / ncta);

    // rows of a group: (segment, first row); gate/up pairs take row n of both matrices. The
    // segments' cumulative group counts come precomputed (no division here).
    auto locate = [&](int grp, int &seg, int &row0) {
        seg = 0;
        row0 = grp;
        if (!GATE_UP) {
            seg = (grp >= p.gend[0]) + (grp >= p.gend[1]);
            row0 = (grp - (seg == 0 ? 0 : p.gend[seg - 1])) * kR;
        }
    };
    auto row_ptr = [&](int seg, int row0, int r, const uint8_t *&cp, const uint16_t *&sp) {
        const DevMatrix &W = GATE_UP ? p.seg[r].W : p.seg[seg].W;
        int row = GATE_UP ? row0 : row0 + r;
        if (row >= W.N) row = (int)W.N - 1;  // masked at the store
        cp = reinterpret_cast<const uint8_t *>(W.codes) + (size_t)row * W.row_bytes;
        sp = Q ? W.scales + (size_t)row * W.scale_stride : nullptr;
    };

    U8 wA[kU][kR], wB[kU][kR];
    float sA[kU][kR][SPC], sB[kU][kR][SPC];
    auto issue = [&](U8 (&wb)[kU][kR], float (&sb)[kU][kR][SPC], int grp, int bat) {
        int seg, row0;
        locate(grp, seg, row0);
#pragma unroll
        for (int r = 0; r < kR; ++r) {
            const uint8_t *cp;
            const uint16_t *sp;
            row_ptr(seg, row0, r, cp, sp);
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int c = (bat * kU + u) * 32 + lane;
                if (c < chunks) {
                    wb[u][r] = ld32(cp + (size_t)c * 32);
                    if (Q) {
#pragma unroll
                        for (int s = 0; s < SPC; ++s) sb[u][r][s] = half_bits_to_float(ld_stream2(sp + c * SPC + s));
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 8; ++k) wb[u][r].w[k] = 0;
#pragma unroll
                    for (int s = 0; s < SPC; ++s) sb[u][r][s] = 0.f;
                }
            }
        }
    };

    // weights do not depend on earlier work: both register buffers are filled before the wait, so
    // that two batches per lane are in flight while the kernels before this one finish (the first
    // step then consumes A without issuing into B). Not for Q4_0 with the post-branch update, whose
    // prologue needs the registers.
    constexpr bool kIssueB = !(PRE && WT == W_Q4_0);
    int grp = g0 + warp, bat = 0;
    bool issued_b = false;
    if (grp < g1) {
        issue(wA, sA, grp, 0);
        int ngrp = grp, nb2 = 1;
        if (nb2 == nbat) { ngrp = grp + kWarps; nb2 = 0; }
        if (kIssueB && ngrp < g1) {
            issue(wB, sB, ngrp, nb2);
            issued_b = true;
        }
    }
    wait();

    // ---- optional post-branch update (x_new = x + t / rms(t) * w): the branch output's 1/rms first
    const int n4 = xs_len / 4;
    float pinv = 0.f;
    if constexpr (PRE) {
        float ts = 0.f;
        for (int i4 = threadIdx.x; i4 < n4 && i4 * 4 < K; i4 += kThreads) {
            const float4 t = __ldcg(reinterpret_cast<const float4 *>(pre.t + i4 * 4));
            ts = fmaf(t.x, t.x, ts);
            ts = fmaf(t.y, t.y, ts);
            ts = fmaf(t.z, t.z, ts);
            ts = fmaf(t.w, t.w, ts);
        }
        ts = warp_sum(ts);
        if (lane == 0) red[warp] = ts;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) tot += red[w];
        pinv = 1.f / sqrtf(tot / (float)K + p.eps);
        __syncthreads();   // red is reused below
    }
    // this CTA's slice of x_new to write (float4 units)
    const int k4 = K / 4, o0 = PRE ? (int)((int64_t)k4 * cta / ncta) : 0, o1 = PRE ? (int)((int64_t)k4 * (cta + 1) / ncta) : 0;

    // ---- stage x (times the norm weight) with independent float4 loads; sum of squares for 1/rms
    float ss = 0.f;
    for (int base = threadIdx.x; base < n4; base += 4 * kThreads) {
        float4 v[4], g[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i4 = base + j * kThreads;
            v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            g[j] = make_float4(1.f, 1.f, 1.f, 1.f);
            if (i4 < n4 && i4 * 4 < K) {
                v[j] = __ldcg(reinterpret_cast<const float4 *>(p.x + i4 * 4));
                if (p.norm_w) g[j] = *reinterpret_cast<const float4 *>(p.norm_w + i4 * 4);
                if constexpr (PRE) {
                    const float4 t = __ldcg(reinterpret_cast<const float4 *>(pre.t + i4 * 4));
                    const float4 w = *reinterpret_cast<const float4 *>(pre.w + i4 * 4);
                    v[j] = make_float4(v[j].x + t.x * pinv * w.x, v[j].y + t.y * pinv * w.y, v[j].z + t.z * pinv * w.z,
                                       v[j].w + t.w * pinv * w.w);
                    if (i4 >= o0 && i4 < o1) *reinterpret_cast<float4 *>(pre.out + i4 * 4) = v[j];
                }
            }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i4 = base + j * kThreads;
            if (i4 >= n4) break;
            ss = fmaf(v[j].x, v[j].x, ss);
            ss = fmaf(v[j].y, v[j].y, ss);
            ss = fmaf(v[j].z, v[j].z, ss);
            ss = fmaf(v[j].w, v[j].w, ss);
            *reinterpret_cast<float4 *>(xs + xs_slot<E>(i4 * 4)) =
                make_float4(v[j].x * g[j].x, v[j].y * g[j].y, v[j].z * g[j].z, v[j].w * g[j].w);
        }
    }
    if (p.norm_w) {
        ss = warp_sum(ss);
        if (lane == 0) red[warp] = ss;
    }
    __syncthreads();
    float inv = 1.f;
    if (p.norm_w) {
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) tot += red[w];
        inv = 1.f / sqrtf(tot / (float)K + p.eps);
    }

    float acc[kR];
#pragma unroll
    for (int r = 0; r < kR; ++r) acc[r] = 0.f;
    // one batch: consume (cw, cs) while the next batch streams into (nw, ns)
    auto step = [&](U8 (&cw)[kU][kR], float (&cs)[kU][kR][SPC], U8 (&nw)[kU][kR], float (&ns)[kU][kR][SPC]) {
        int ngrp = grp, nb2 = bat + 1;
        if (nb2 == nbat) { ngrp = grp + kWarps; nb2 = 0; }
        if (ngrp < g1 && !issued_b) issue(nw, ns, ngrp, nb2);
        issued_b = false;
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int s = bat * kU + u;
            if (s < slabs) {
                const float *xp = xs + s * 32 * E + lane * 4;
#pragma unroll
                for (int r = 0; r < kR; ++r) {
                    if constexpr (WT == W_Q4_0) {
                        const float2 d = Chunk32<W_Q4_0>::dot2(cw[u][r], xp);
                        acc[r] = fmaf(cs[u][r][0], d.x, acc[r]);
                        acc[r] = fmaf(cs[u][r][SPC - 1], d.y, acc[r]);
                    } else if constexpr (WT == W_Q8_0) {
                        acc[r] = fmaf(cs[u][r][0], Chunk32<W_Q8_0>::dot(cw[u][r], xp), acc[r]);
                    } else {
                        acc[r] += Chunk32<WT>::dot(cw[u][r], xp);
                    }
                }
            }
        }
        if (nb2 == 0) {
            // the row pair is done: reduce across the warp and apply the epilogue
#pragma unroll
            for (int r = 0; r < kR; ++r) acc[r] = warp_sum(acc[r]) * inv;
            if (lane == 0) {
                int seg, row0;
                locate(grp, seg, row0);
                if (GATE_UP) {
                    float gv = acc[0], uv = acc[1];
                    if (p.seg[0].bias) gv += p.seg[0].bias[row0];
                    if (p.seg[1].bias) uv += p.seg[1].bias[row0];
                    p.seg[0].out[row0] = apply_act(p.act, gv) * uv;
                } else {
                    const GemvSeg &S = p.seg[seg];
#pragma unroll
                    for (int r = 0; r < kR; ++r) {
                        if (row0 + r >= S.W.N) continue;
                        float y = acc[r];
                        if (S.bias) y += S.bias[row0 + r];
                        if (S.epi == EPI_ADD) y += __ldcg(S.out + row0 + r);
                        S.out[row0 + r] = y;
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < kR; ++r) acc[r] = 0.f;
        }
        grp = ngrp;
        bat = nb2;
        return grp < g1;
    };
    if (grp < g1) {
        while (step(wA, sA, wB, sB) && step(wB, sB, wA, sA)) {
        }
    }
    __syncthreads();  // xs and red are reused by whatever runs next in this CTA
}


template <int WT> inline size_t gemv_smem_bytes(size_t row_bytes) {
    const int chunks = (int)(row_bytes / 32);
    const int slabs = (chunks + 31) / 32;
    return (size_t)slabs * 32 * Chunk32<WT>::E * sizeof(float);
}

inline size_t gemv_smem_bytes_rt(int wtype, size_t row_bytes) {
    switch (wtype) {
    case W_F32: return gemv_smem_bytes<W_F32>(row_bytes);
    case W_F16: return gemv_smem_bytes<W_F16>(row_bytes);
    case W_Q8_0: return gemv_smem_bytes<W_Q8_0>(row_bytes);
    default: return gemv_smem_bytes<W_Q4_0>(row_bytes);
    }
}

inline int gemv_groups(const GemvParams &p, int kr) {
    if (p.gate_up) return (int)p.seg[0].W.N;
    int groups = 0;
    for (int i = 0; i < p.nseg; ++i) groups += (int)((p.seg[i].W.N + kr - 1) / kr);
    return groups;
}

}  // namespace syn
