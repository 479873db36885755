// Device bodies of the row preparation, the attention combine and the
// acceptance step, shared by their per-launch kernels and the persistent
// round kernel.
#pragma once

#include "gemm.cuh"
#include "kernels.cuh"

namespace dfl {
namespace kdev {

constexpr int COMBINE_MAXC = 512;   // chunks one combine folds (32768 keys)

// Key range [lo, hi) the forward's rows attend and its row count / position.
__device__ __forceinline__ void attn_range(const AttnArgs& a, int* lo, int* hi, int* T, int* pos0) {
    *T = a.st->fwd_T;
    *pos0 = a.st->fwd_pos0;
    *hi = *pos0 + *T;
    *lo = (!a.causal && a.window > 0) ? max(0, *pos0 - a.window) : 0;
}

// Row t of a forward: sets the forward descriptor (row 0's caller also
// writes it to the device state), gathers the embedding row into the fp32
// residual, writes layer 0's folded-norm input and the RoPE angles.  Run by
// nthr threads (tid 0..nthr-1) that share sh[3] and the barrier bar().
template <class Bar>
__device__ __forceinline__ void prepare_row(const RowsArgs& a, int t, int tid, int nthr,
                                            volatile int* sh, Bar bar) {
    DevState* st = a.st;
    if (tid == 0) {
        int T = 0, pos0 = 0;
        if (a.mode == FWD_PREFILL) {
            T = a.T;
            pos0 = a.pos0;
        } else if (!st->finished) {
            pos0 = st->n;
            if (a.mode == FWD_DRAFT) T = st->bl > 1 ? st->bl : 0;
            else if (a.mode == FWD_VERIFY) T = st->bl;
            else T = 1;   // FWD_GREEDY
        }
        int tok = 0;
        if (t < T) {
            if (a.mode == FWD_PREFILL) tok = a.tokens ? a.tokens[pos0 + t] : 0;
            else if (t == 0) tok = st->t_n;
            else if (a.mode == FWD_DRAFT) tok = a.mask_id;
            else tok = a.tokens[t - 1];
            if (tok < 0 || tok >= a.vocab) {
                set_error(st, DERR_TOKEN, tok);
                tok = 0;
            }
        }
        sh[0] = T;
        sh[1] = pos0;
        sh[2] = tok;
        if (t == 0) {
            st->fwd_T = T;
            st->fwd_pos0 = pos0;
            st->fwd_commit = 0;
            st->fwd_commit_r0 = 0;
            if (a.mode == FWD_DRAFT) st->draft_bl = T;
        }
        if (a.amax) a.amax[t] = 0ull;
    }
    bar();
    const int T = sh[0];
    float* xr = a.x + (size_t)t * a.hidden;
    if (t < T && a.embed) {
        for (int i = tid; i < a.hidden; i += nthr) {
            const size_t e = (size_t)sh[2] * a.hidden + i;
            xr[i] = a.embed_f32 ? reinterpret_cast<const float*>(a.embed)[e]
                                : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.embed)[e]);
        }
    } else if (t < T && a.x_src) {
        for (int i = tid; i < a.hidden; i += nthr) xr[i] = a.x_src[(size_t)t * a.hidden + i];
    } else if (a.embed || a.x_src) {
        for (int i = tid; i < a.hidden; i += nthr) xr[i] = 0.f;
    }
    if (a.embed || a.x_src) {
        // folded RMSNorm input of the next matrix (layer 0's, or with x_src
        // the final norm's): xn = x * w0, per-128-column sums of x^2
        bar();
        for (int i = tid; i < a.hidden; i += nthr)
            store_act(a.xn, a.xn_type, a.hidden, t, i, xr[i] * a.w0[i]);
        const int warp = tid >> 5, lane = tid & 31;
        for (int b = warp; b < a.hidden / 128; b += nthr >> 5) {
            float ss = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float v = xr[b * 128 + lane * 4 + j];
                ss = fmaf(v, v, ss);
            }
            ss = warp_sum(ss);
            if (lane == 0) a.ssq[b * DFL_MAX_ROWS + t] = ss;
        }
    }
    // the row's RoPE angles from the position table (made once at init by
    // rope_rows_kernel: pos * theta^(-2i/d) in double, reduced with a
    // two-part 2 pi, cos / sin in double, rounded once to fp32); a row past
    // the table (never one the forward uses) gets the identity rotation
    const int half = a.head_dim / 2, pos = sh[1] + t;
    const bool in_tab = pos >= 0 && pos < a.tab_rows;
    for (int i = tid; i < half; i += nthr) {
        a.rope_cos[t * half + i] = in_tab ? a.tab_cos[(size_t)pos * half + i] : 1.f;
        a.rope_sin[t * half + i] = in_tab ? a.tab_sin[(size_t)pos * half + i] : 0.f;
    }
}

// Folds the chunks of one (row, q head) in chunk order and normalises.  The
// chunk maxima and sums are staged in shared memory by all threads at once;
// every thread then folds its output element over the chunks in chunk
// order (fully masked chunks add exact zeros at the end, so a row's result
// does not depend on the forward's row count).
// One (q head hq, row t) item run by HD threads (d = 0..HD-1) sharing
// s_w / s_l [COMBINE_MAXC], s_red [HD/32] and the barrier bar().
template <int HD, class Bar>
__device__ __forceinline__ void combine_item(const AttnArgs& a, int hq, int t, int d, float* s_w,
                                             float* s_l, float* s_red, Bar bar) {
    constexpr int MAXC = COMBINE_MAXC;
    int lo, hi, T, pos0;
    attn_range(a, &lo, &hi, &T, &pos0);
    const size_t ld = (size_t)a.n_q * HD, col = (size_t)hq * HD + d;
    if (t >= T) {
        store_act(a.out, a.out_type, ld, t, col, 0.f);
        return;
    }
    const int c_lo = lo / ATTN_CHUNK, c_hi = (hi - 1) / ATTN_CHUNK;
    const int nc = c_hi - c_lo + 1;
    const size_t cstride = (size_t)DFL_MAX_ROWS * a.n_q * (HD + 2);
    const float* base = a.part + ((size_t)c_lo * DFL_MAX_ROWS + t) * a.n_q * (HD + 2) +
                        (size_t)hq * (HD + 2);
    if (nc > MAXC) {
        if (d == 0) set_error(a.st, DERR_INDEX, nc);
        return;
    }
    float mx = -INFINITY;
    for (int i = d; i < nc; i += HD) {
        const float m = base[i * cstride];
        s_w[i] = m;
        s_l[i] = base[i * cstride + 1];
        mx = fmaxf(mx, m);
    }
    mx = warp_max(mx);
    if ((d & 31) == 0) s_red[d >> 5] = mx;
    bar();
    float M = s_red[0];
#pragma unroll
    for (int w = 1; w < HD / 32; ++w) M = fmaxf(M, s_red[w]);
    for (int i = d; i < nc; i += HD) s_w[i] = (s_w[i] == -INFINITY) ? 0.f : expf(s_w[i] - M);
    bar();
    float L = 0.f, O = 0.f;
    int i = 0;
    for (; i + 4 <= nc; i += 4) {
        const float o0 = base[(i + 0) * cstride + 2 + d], o1 = base[(i + 1) * cstride + 2 + d];
        const float o2 = base[(i + 2) * cstride + 2 + d], o3 = base[(i + 3) * cstride + 2 + d];
        O = fmaf(o0, s_w[i + 0], O);
        O = fmaf(o1, s_w[i + 1], O);
        O = fmaf(o2, s_w[i + 2], O);
        O = fmaf(o3, s_w[i + 3], O);
    }
    for (; i < nc; ++i) O = fmaf(base[i * cstride + 2 + d], s_w[i], O);
    for (int j = 0; j < nc; ++j) L = fmaf(s_l[j], s_w[j], L);
    store_act(a.out, a.out_type, ld, t, col, O / L);
}

// Acceptance and round bookkeeping from the forward's packed argmax keys
// (one thread).
__device__ __forceinline__ void accept_run(const AcceptArgs& a) {
    DevState* st = a.st;
    const int T = st->fwd_T;
    int y[DFL_MAX_ROWS];
    for (int i = 0; i < DFL_MAX_ROWS; ++i) y[i] = argmax_key_index(a.amax[i]);
    if (a.mode == FWD_DRAFT) {
        for (int j = 0; j < a.block_max - 1; ++j)
            a.draft_out[j] = (j + 1 < T) ? y[j + 1] : -1;
        return;
    }
    const int B = a.block_max;
    if (a.mode == FWD_PREFILL) {
        st->t_n = y[T - 1];
        st->n = a.prompt_len;
        st->generated = 1;
        st->max_new = a.max_new;
        st->ctx_len = a.prompt_len;
        st->rounds = 0;
        st->emitted = 0;
        for (int j = 0; j < 16; ++j) st->accept_hist[j] = 0;
        st->last_a = 0;
        st->finished = (a.eos_id >= 0 && st->t_n == a.eos_id) || a.max_new <= 1 ||
                       st->n >= a.max_seq;
        st->acc_ema = (float)(B - 1);
        const int bl = min(block_cap(st, B), min(a.max_new - 1, a.max_seq - st->n));
        st->bl = st->finished ? 0 : bl;
        return;
    }
    // VERIFY / GREEDY
    if (T == 0) {
        *a.n_emitted = 0;
        for (int j = 0; j < B; ++j) a.tokens_out[j] = -1;
        st->fwd_commit = 0;
        return;
    }
    int acc = 0;
    if (a.mode == FWD_VERIFY)
        while (acc < T - 1 && a.draft_ids[acc] == y[acc]) ++acc;
    int emit = acc + 1;
    int fin = 0;
    if (a.eos_id >= 0) {
        for (int i = 0; i <= acc; ++i)
            if (y[i] == a.eos_id) {
                emit = i + 1;
                fin = 1;
                break;
            }
    }
    for (int j = 0; j < B; ++j) a.tokens_out[j] = j < emit ? y[j] : -1;
    *a.n_emitted = emit;
    const int n_old = st->n;
    st->n = n_old + emit;
    st->t_n = y[emit - 1];
    st->generated += emit;
    st->ctx_len = st->n;
    st->rounds += 1;
    st->emitted += emit;
    for (int j = 0; j < acc && j < 16; ++j) st->accept_hist[j] += 1;
    st->last_a = acc;
    st->acc_ema = 0.5f * st->acc_ema + 0.5f * (float)acc;
    fin |= st->generated >= st->max_new || st->n >= a.max_seq;
    st->finished = fin;
    st->bl = fin ? 0 : min(block_cap(st, B), min(st->max_new - st->generated, a.max_seq - st->n));
    st->fwd_commit_r0 = 0;
    st->fwd_commit = emit;
}

}  // namespace kdev
}  // namespace dfl
