// Non-GEMM kernels of the DFlash round: row preparation (embedding gather,
// RoPE angles), RMSNorm, per-head q/k norm + RoPE + KV-cache write, split-KV
// attention with a fixed chunk size, acceptance / rollback bookkeeping, the
// hc-stream tap reduce and the INT4 group-64 quantiser.
//
// By page: the block [t_n, MASK...] drafted in one forward ("[RFC] DFlash",
// "DFlash Overview"); first-mismatch acceptance with the bonus token and
// KV-cache position rollback ("[RFC] DFlash", "Key Implementation Details",
// Phase 3), the dynamic block length ("Requested changes" 1), EOS keeping
// the first EOS (the second review); the per-token mean over the
// hyper-connection streams ("dflash: the chain verify builds pipelined ...",
// first commit); projections quantised to INT4 at load ("feat: DFlash2
// block-diffusion drafter for Qwen 3.8", third commit), here the group-64
// symmetric format with bf16 scales of the long-context drafter workload.
//
// All kernels read the forward's row count and position from the device
// state, so a round needs no host round-trip; rows beyond the forward's
// count are written as zeros, which keeps every padded GEMM column zero.

#include "kernels_dev.cuh"
#include "rows_dev.cuh"

namespace dfl {

namespace {

__device__ __forceinline__ float ld_any(const void* base, int t, size_t i) {
    if (t == XT_F32) return reinterpret_cast<const float*>(base)[i];
    if (t == XT_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[i]);
    return __half2float(reinterpret_cast<const __half*>(base)[i]);
}

// --------------------------------------------------------------- prepare rows

// One CTA: sets the forward descriptor (thread 0), then every CTA gathers
// its row of the embedding into the fp32 residual and fills the RoPE table.
struct BlockBar {
    __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

// One CTA per row (see kdev::prepare_row).
__global__ void prepare_rows_kernel(RowsArgs a) {
    pdl_trigger();
    pdl_wait();
    __shared__ int sh[3];
    kdev::prepare_row(a, blockIdx.x, threadIdx.x, blockDim.x, sh, BlockBar());
}

// --------------------------------------------------------------- attention

using kdev::attn_range;

// One CTA per (kv head, chunk of ATTN_CHUNK keys): partial softmax state
// (max m, sum l, unnormalised output o) of every query row of the kv head's
// query-head group.  Keys outside the range, or after the query under the
// causal rule, weigh exactly zero.
template <int HD>
__global__ void attn_partial_kernel(AttnArgs a) {
    pdl_trigger();
    pdl_wait();
    constexpr int C = ATTN_CHUNK;
    const int kh = blockIdx.x, c = blockIdx.y;
    int lo, hi, T, pos0;
    attn_range(a, &lo, &hi, &T, &pos0);
    if (T == 0) return;
    const int k0 = c * C;
    if (k0 >= hi || k0 + C <= lo) return;
    extern __shared__ float sm[];
    float* Ks = sm;                    // [C][HD]
    float* Vs = Ks + C * HD;           // [C][HD]
    float* Ps = Vs + C * HD;           // [warps][C]
    float* Qs = Ps + (blockDim.x >> 5) * C;   // [warps][HD]
    const int group = a.n_q / a.n_kv;
    const size_t kbase = (size_t)kh * a.cap * HD;
    for (int e = threadIdx.x; e < C * HD; e += blockDim.x) {
        const int j = e / HD, d = e % HD;
        const int key = k0 + j;
        const bool in = key >= lo && key < hi;
        Ks[e] = in ? ld_any(a.k_cache, a.kv_type, kbase + (size_t)key * HD + d) : 0.f;
        Vs[e] = in ? ld_any(a.v_cache, a.kv_type, kbase + (size_t)key * HD + d) : 0.f;
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, warps = blockDim.x >> 5;
    const int nq = group * T;
    for (int qi = warp; qi < nq; qi += warps) {
        const int hq = kh * group + qi / T, t = qi % T;
        const size_t qoff = ((size_t)hq * DFL_MAX_ROWS + t) * HD;   // [n_q][16][HD]
        for (int d = lane; d < HD; d += 32) Qs[warp * HD + d] = ld_any(a.q, a.kv_type, qoff + d);
        __syncwarp();
        float s[C / 32];
        bool valid[C / 32];
        float m = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < C / 32; ++jj) {
            const int j = lane + 32 * jj, key = k0 + j;
            float acc = 0.f;
            for (int d = 0; d < HD; ++d) acc = fmaf(Qs[warp * HD + d], Ks[j * HD + d], acc);
            s[jj] = acc * a.scale;
            valid[jj] = key >= lo && key < hi && (!a.causal || key <= pos0 + t);
            if (valid[jj]) m = fmaxf(m, s[jj]);
        }
        m = warp_max(m);
        float l = 0.f;
#pragma unroll
        for (int jj = 0; jj < C / 32; ++jj) {
            const float p = valid[jj] ? expf(s[jj] - m) : 0.f;
            Ps[warp * C + lane + 32 * jj] = p;
            l += p;
        }
        l = warp_sum(l);
        __syncwarp();
        float* dst = a.part + (((size_t)c * DFL_MAX_ROWS + t) * a.n_q + hq) * (HD + 2);
        for (int d = lane; d < HD; d += 32) {
            float o = 0.f;
            for (int j = 0; j < C; ++j) o = fmaf(Ps[warp * C + j], Vs[j * HD + d], o);
            dst[2 + d] = o;
        }
        if (lane == 0) {
            dst[0] = m;
            dst[1] = l;
        }
        __syncwarp();
    }
}

// One CTA per (q head, row) (see kdev::combine_item).
template <int HD>
__global__ void attn_combine_kernel(AttnArgs a) {
    pdl_trigger();
    pdl_wait();
    __shared__ float s_w[kdev::COMBINE_MAXC];
    __shared__ float s_l[kdev::COMBINE_MAXC];
    __shared__ float s_red[HD / 32];
    kdev::combine_item<HD>(a, blockIdx.x, blockIdx.y, threadIdx.x, s_w, s_l, s_red, BlockBar());
}

// --------------------------------------------------------------- acceptance

__global__ void accept_kernel(AcceptArgs a) {
    pdl_trigger();
    pdl_wait();
    if (threadIdx.x == 0) kdev::accept_run(a);
}

__global__ void set_chunk_kernel(DevState* st, int pos0, int T, int commit_lo) {
    pdl_trigger();
    pdl_wait();
    st->fwd_pos0 = pos0;
    st->fwd_T = T;
    const int r0 = max(0, commit_lo - pos0);
    st->fwd_commit_r0 = min(r0, T);
    st->fwd_commit = max(0, T - st->fwd_commit_r0);
}

__global__ void rollback_kernel(DevState* st, int new_len, int token, int B, int max_seq) {
    pdl_trigger();
    pdl_wait();
    const int old = st->n;
    st->n = new_len;
    st->t_n = token;
    if (st->ctx_len > new_len) st->ctx_len = new_len;
    st->generated = max(1, st->generated - (old - new_len));
    st->finished = st->generated >= st->max_new || new_len >= max_seq;
    st->bl = st->finished ? 0 : min(block_cap(st, B), min(st->max_new - st->generated, max_seq - new_len));
}

__global__ void set_ext_state_kernel(DevState* st, int n_ext, int tok, int max_new, int B,
                                     int max_seq, int eos) {
    pdl_trigger();
    pdl_wait();
    st->n = n_ext;
    st->t_n = tok;
    st->generated = 1;
    st->max_new = max_new;
    st->ctx_len = n_ext;
    st->rounds = 0;
    st->emitted = 0;
    for (int j = 0; j < 16; ++j) st->accept_hist[j] = 0;
    st->last_a = 0;
    st->finished = (eos >= 0 && tok == eos) || max_new <= 1 || n_ext >= max_seq;
    st->acc_ema = (float)(B - 1);
    st->bl = st->finished ? 0 : min(block_cap(st, B), min(max_new - 1, max_seq - n_ext));
    st->fwd_T = 0;
    st->fwd_commit = 0;
}

// --------------------------------------------------------------- tap reduce

// out[r][i*H + j] = (1/hc) * sum_{s=0..hc-1} src_i[r][s*H + j]; eight
// consecutive columns per thread (16-byte loads of bf16 streams).
template <typename IT, typename OT, bool SPLIT = false>
__global__ void tap_reduce_kernel(TapArgs a) {
    pdl_trigger();
    pdl_wait();
    const long long per_row = (long long)a.n_layers * a.hidden / 8;
    const long long total = per_row * a.rows;
    const float inv = 1.0f / (float)a.hc;
    for (long long v = (long long)blockIdx.x * blockDim.x + threadIdx.x; v < total;
         v += (long long)gridDim.x * blockDim.x) {
        const int r = (int)(v / per_row);
        const int col = (int)(v % per_row) * 8;
        const int layer = col / a.hidden, j = col % a.hidden;
        const IT* src = reinterpret_cast<const IT*>(a.src[layer]) +
                        (size_t)r * a.hc * a.hidden + j;
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        for (int s = 0; s < a.hc; ++s) {
            if (sizeof(IT) == 2) {
                const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src + (size_t)s * a.hidden));
                const IT* p = reinterpret_cast<const IT*>(&raw);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] += to_f32<IT>(p[e]);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] += to_f32<IT>(src[(size_t)s * a.hidden + e]);
            }
        }
        OT* dst = reinterpret_cast<OT*>(a.out) + (size_t)r * a.out_row_stride + col;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float v = acc[e] * inv;
            const OT hi = from_f32<OT>(v);
            dst[e] = hi;
            // XT_BF16S: the rounding remainder 16 rows further down, or lo_offset away
            if (SPLIT)
                dst[e + (a.lo_offset ? a.lo_offset : DFL_MAX_ROWS * a.out_row_stride)] =
                    from_f32<OT>(v - to_f32<OT>(hi));
        }
    }
}

// --------------------------------------------------------------- window ingest

// One CTA of 256 threads per row: sum of squares in a fixed order (per
// thread, then the warp tree, then the warps in order), then the row.
__global__ void ctx_rows_kernel(CtxRowsArgs a) {
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.x, tid = threadIdx.x;
    const float* y = a.y + (size_t)r * a.hidden;
    __shared__ float s_part[8];
    float rstd = 1.f;
    if (a.norm) {
        float ss = 0.f;
        for (int j = tid; j < a.hidden; j += 256) ss = fmaf(y[j], y[j], ss);
        ss = warp_sum(ss);
        if ((tid & 31) == 0) s_part[tid >> 5] = ss;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) tot += s_part[w];
        rstd = 1.0f / sqrtf(tot / (float)a.hidden + a.eps);
    }
    for (int j = tid; j < a.hidden; j += 256) {
        const float v = a.norm ? y[j] * a.w[j] * rstd : y[j];
        const size_t i = (size_t)r * a.hidden + j;
        if (a.f16) {
            const __half h = __float2half_rn(v);
            reinterpret_cast<__half*>(a.c_hi)[i] = h;
            reinterpret_cast<__half*>(a.c_lo)[i] = __float2half_rn(v - __half2float(h));
        } else {
            const __nv_bfloat16 h = __float2bfloat16_rn(v);
            reinterpret_cast<__nv_bfloat16*>(a.c_hi)[i] = h;
            reinterpret_cast<__nv_bfloat16*>(a.c_lo)[i] = __float2bfloat16_rn(v - __bfloat162float(h));
        }
    }
}

// ---- dense prompt prefill

__global__ void embed_rows_kernel(const int32_t* tokens, int rows, const __nv_bfloat16* embed, int hidden,
                                  int vocab, float* x, DevState* st) {
    pdl_trigger();
    pdl_wait();
    const int r = blockIdx.x;
    int tok = tokens[r];
    if (tok < 0 || tok >= vocab) {
        if (threadIdx.x == 0) set_error(st, DERR_TOKEN, tok);
        tok = -1;
    }
    for (int j = threadIdx.x; j < hidden; j += blockDim.x)
        x[(size_t)r * hidden + j] = tok < 0 ? 0.f : __bfloat162float(embed[(size_t)tok * hidden + j]);
}

// One CTA of RN_THREADS threads per row; sum of squares in a fixed order.
// A thread holds its (up to RN_PER) elements of the row in registers: all
// of its loads, every split-K slab's included, are issued before the first
// use, instead of one round trip per element or slab (rows wider than
// RN_THREADS x RN_PER = 4096 take the plain loop).
constexpr int RN_THREADS = 512, RN_PER = 8;
__device__ __forceinline__ void resid_norm_row(const ResidNormArgs& a) {
    pdl_trigger();
    pdl_wait();
    constexpr int PER = RN_PER, NT = RN_THREADS;
    const int r = blockIdx.x, tid = threadIdx.x;
    float* x = a.x + (size_t)r * a.hidden;
    const float* y = a.y ? a.y + (size_t)r * a.hidden : nullptr;
    __shared__ float s_part[NT / 32];
    float ss = 0.f;
    float v[PER];
    const bool held = a.hidden <= NT * PER;
    if (held) {
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int j = tid + NT * i;
            v[i] = j < a.hidden ? x[j] : 0.f;
        }
        if (y) {
            float w[PER];
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int j = tid + NT * i;
                w[i] = j < a.hidden ? y[j] : 0.f;
            }
            if (a.y_splits > 1) {
                // every split's loads of 8 columns in flight at once, then
                // the adds in split order (a split at a time cost one L2
                // round trip per split)
#pragma unroll
                for (int i0 = 0; i0 < PER; i0 += 8) {
                    float u[7][8];
#pragma unroll
                    for (int z = 1; z < 8; ++z)
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int j = tid + NT * (i0 + i);
                            u[z - 1][i] = (z < a.y_splits && j < a.hidden)
                                              ? __ldcg(y + (size_t)z * a.y_slab + j) : 0.f;
                        }
#pragma unroll
                    for (int z = 1; z < 8; ++z)
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            if (z < a.y_splits) w[i0 + i] += u[z - 1][i];
                }
                for (int z = 8; z < a.y_splits; ++z)
#pragma unroll
                    for (int i = 0; i < PER; ++i) {
                        const int j = tid + NT * i;
                        if (j < a.hidden) w[i] += __ldcg(y + (size_t)z * a.y_slab + j);
                    }
            }
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int j = tid + NT * i;
                v[i] += w[i];
                if (j < a.hidden) x[j] = v[i];
            }
        }
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int j = tid + NT * i;
            if (j < a.hidden) {
                if (a.tap_hi) store_hilo(a.tap_hi, a.tap_lo, (size_t)r * a.tap_ld + a.tap_col + j, v[i]);
                ss = fmaf(v[i], v[i], ss);
            }
        }
    } else {
        for (int j = tid; j < a.hidden; j += NT) {
            float u = x[j];
            if (y) {
                float t = y[j];
                for (int z = 1; z < a.y_splits; ++z) t += __ldcg(y + (size_t)z * a.y_slab + j);
                u += t;
                x[j] = u;
            }
            if (a.tap_hi) store_hilo(a.tap_hi, a.tap_lo, (size_t)r * a.tap_ld + a.tap_col + j, u);
            ss = fmaf(u, u, ss);
        }
    }
    ss = warp_sum(ss);
    if ((tid & 31) == 0) s_part[tid >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) tot += s_part[w];
    const float rstd = 1.0f / sqrtf(tot / (float)a.hidden + a.eps);
    if (held) {
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int j = tid + NT * i;
            if (j < a.hidden) store_hilo(a.hi, a.lo, (size_t)r * a.hidden + j, v[i] * a.w[j] * rstd, a.f16);
        }
    } else {
        for (int j = tid; j < a.hidden; j += NT)
            store_hilo(a.hi, a.lo, (size_t)r * a.hidden + j, x[j] * a.w[j] * rstd, a.f16);
    }
}

__global__ void __launch_bounds__(RN_THREADS) resid_norm_kernel(ResidNormArgs a) { resid_norm_row(a); }

// The same row for the many rows of a dense pass, with the registers capped
// so that two CTAs share an SM (at one CTA per SM the kernel waits on its
// loads).
__global__ void __launch_bounds__(RN_THREADS, 2) resid_norm_wide_kernel(ResidNormArgs a) { resid_norm_row(a); }

// One warp per (row, head) over the q, k and v heads; lane l holds
// elements l + 32 m (rotate-half pairs m with m + per/2 in the same lane).
__global__ void qkv_rows_kernel(QkvRowsArgs a) {
    pdl_trigger();
    pdl_wait();
    const int heads = a.n_q + 2 * a.n_kv;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (warp >= a.rows * heads) return;
    const int r = warp / heads, h = warp % heads;
    const bool is_q = h < a.n_q, is_k = !is_q && h < a.n_q + a.n_kv;
    const int hd = a.head_dim, per = hd / 32;
    const int pos = a.pos0 + r;
    const float* src = a.y + (size_t)r * heads * hd + (size_t)h * hd;
    float v[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) v[m] = m < per ? src[lane + 32 * m] : 0.f;
    if (is_q || is_k) {
        const float* nw = is_q ? a.q_norm : a.k_norm;
        float ss = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) ss = fmaf(v[m], v[m], ss);
        ss = warp_sum(ss);
        const float inv = 1.0f / sqrtf(ss / (float)hd + a.eps);
#pragma unroll
        for (int m = 0; m < 4; ++m) v[m] = m < per ? v[m] * inv * nw[lane + 32 * m] : 0.f;
        float cs[2], sn[2];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            cs[m] = 1.f;
            sn[m] = 0.f;
            if (m < per / 2) {
                cs[m] = a.rope_cos[(size_t)r * (hd / 2) + lane + 32 * m];
                sn[m] = a.rope_sin[(size_t)r * (hd / 2) + lane + 32 * m];
            }
        }
        float o[4];
        if (per == 4) {
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                o[m] = v[m] * cs[m] - v[m + 2] * sn[m];
                o[m + 2] = v[m + 2] * cs[m] + v[m] * sn[m];
            }
        } else {
            o[0] = v[0] * cs[0] - v[1] * sn[0];
            o[1] = v[1] * cs[0] + v[0] * sn[0];
            o[2] = o[3] = 0.f;
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) v[m] = o[m];
    }
    if (is_q) {
        __half* q = reinterpret_cast<__half*>(a.q_out) +
                    (((size_t)(r >> 4) * a.n_q + h) * DFL_MAX_ROWS + (r & 15)) * hd;
#pragma unroll
        for (int m = 0; m < 4; ++m)
            if (m < per) q[lane + 32 * m] = __float2half_rn(v[m]);
        return;
    }
    if (pos < 0 || pos >= a.max_seq || pos >= a.cap) {
        if (lane == 0) set_error(a.st, DERR_INDEX, pos);
        return;
    }
    const int kh = is_k ? h - a.n_q : h - a.n_q - a.n_kv;
    void* cache = is_k ? a.k_cache : a.v_cache;
    const size_t base = ((size_t)kh * a.cap + pos) * hd;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        if (m >= per) continue;
        const size_t i = base + lane + 32 * m;
        if (a.c_type == XT_F32) reinterpret_cast<float*>(cache)[i] = v[m];
        else if (a.c_type == XT_BF16) reinterpret_cast<__nv_bfloat16*>(cache)[i] = __float2bfloat16_rn(v[m]);
        else reinterpret_cast<__half*>(cache)[i] = __float2half_rn(v[m]);
    }
}

__global__ void rope_rows_kernel(int pos0, int rows, int half, const double* inv_freq, float* cs,
                                 float* sn) {
    pdl_trigger();
    pdl_wait();
    const long long n = (long long)rows * half;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (long long)gridDim.x * blockDim.x) {
        const int r = (int)(e / half), i = (int)(e % half);
        const double ang = (double)(pos0 + r) * inv_freq[i];
        const double k = rint(ang * 0.15915494309189535);
        double rr = fma(-k, 6.283185307179586, ang);
        rr = fma(-k, 2.4492935982947064e-16, rr);
        cs[e] = (float)cos(rr);
        sn[e] = (float)sin(rr);
    }
}

// One thread per 32-bit word of the packed rows (8 consecutive inputs).
__global__ void dequant_int4g64_f16_kernel(const uint32_t* __restrict__ packed,
                                           const uint16_t* __restrict__ scales, int n, int k,
                                           __half* __restrict__ out) {
    pdl_trigger();
    pdl_wait();
    const long long words = (long long)n * (k / 8);
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < words;
         i += (long long)gridDim.x * blockDim.x) {
        const int row = (int)(i / (k / 8)), k0 = (int)(i % (k / 8)) * 8;
        const uint32_t wv = packed[i];
        const float sc = __uint_as_float((uint32_t)scales[(size_t)(k0 / 64) * n + row] << 16);
        __half h[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            h[2 * j] = __float2half_rn((float)((int)((wv >> (4 * j)) & 15u) - 8) * sc);
            h[2 * j + 1] = __float2half_rn((float)((int)((wv >> (4 * j + 16)) & 15u) - 8) * sc);
        }
        *reinterpret_cast<uint4*>(out + (size_t)row * k + k0) = *reinterpret_cast<const uint4*>(h);
    }
}

// One warp per (row, kv head, K or V); lane l holds elements l + 32 m.
__global__ void ctx_kv_store_kernel(CtxKvArgs a) {
    pdl_trigger();
    pdl_wait();
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    const int items = a.rows * a.n_kv * 2;
    if (warp >= items) return;
    const int r = warp / (2 * a.n_kv), rem = warp % (2 * a.n_kv);
    const bool is_k = rem < a.n_kv;
    const int kh = is_k ? rem : rem - a.n_kv;
    const int hd = a.head_dim, per = hd / 32;
    const int pos = a.pos0 + r;
    if (pos < 0 || pos >= a.max_seq || pos >= a.cap) {
        if (lane == 0) set_error(a.st, DERR_INDEX, pos);
        return;
    }
    const float* src = a.y + (size_t)r * 2 * a.n_kv * hd + (size_t)rem * hd;
    float v[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) v[m] = m < per ? src[lane + 32 * m] : 0.f;
    if (is_k) {
        float ss = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) ss = fmaf(v[m], v[m], ss);
        ss = warp_sum(ss);
        const float inv = 1.0f / sqrtf(ss / (float)hd + a.eps);
#pragma unroll
        for (int m = 0; m < 4; ++m) v[m] = m < per ? v[m] * inv * a.k_norm[lane + 32 * m] : 0.f;
        // rotate-half RoPE at `pos`: element i pairs with i + hd/2 (m and m + per/2)
        float cs[2], sn[2];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            cs[m] = 1.f;
            sn[m] = 0.f;
            if (m < per / 2) {
                cs[m] = a.rope_cos[(size_t)r * (hd / 2) + lane + 32 * m];
                sn[m] = a.rope_sin[(size_t)r * (hd / 2) + lane + 32 * m];
            }
        }
        float o[4];
        if (per == 4) {
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                o[m] = v[m] * cs[m] - v[m + 2] * sn[m];
                o[m + 2] = v[m + 2] * cs[m] + v[m] * sn[m];
            }
        } else {
            o[0] = v[0] * cs[0] - v[1] * sn[0];
            o[1] = v[1] * cs[0] + v[0] * sn[0];
            o[2] = o[3] = 0.f;
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) v[m] = o[m];
    }
    void* cache = is_k ? a.k_cache : a.v_cache;
    const size_t base = ((size_t)kh * a.cap + pos) * hd;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
        if (m >= per) continue;
        const size_t i = base + lane + 32 * m;
        if (a.c_type == XT_F32) reinterpret_cast<float*>(cache)[i] = v[m];
        else if (a.c_type == XT_BF16) reinterpret_cast<__nv_bfloat16*>(cache)[i] = __float2bfloat16_rn(v[m]);
        else reinterpret_cast<__half*>(cache)[i] = __float2half_rn(v[m]);
    }
}

// --------------------------------------------------------------- INT4 quantiser

// One warp per (row, 256 consecutive k): lane holds 8 consecutive values;
// lanes 8q..8q+7 form group q.
__global__ void quantize_int4g64_kernel(const float* __restrict__ w, int n, int k,
                                        uint8_t* __restrict__ packed, uint16_t* __restrict__ scales) {
    pdl_trigger();
    pdl_wait();
    const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int per_row = k / 256;
    if (gw >= n * per_row) return;
    const int row = gw / per_row, kb = gw % per_row;
    const int k0 = kb * 256 + lane * 8;
    const float* src = w + (size_t)row * k + k0;
    float v[8];
    float am = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        v[e] = src[e];
        am = fmaxf(am, fabsf(v[e]));
    }
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    const __nv_bfloat16 sb = __float2bfloat16_rn(__fdiv_rn(am, 7.0f));
    const float s = __bfloat162float(sb);
    // interleaved word: k0+2j at nibble j, k0+2j+1 at nibble j+4 (j = 0..3)
    uint32_t word = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        int q = 0;
        if (s > 0.f) {
            q = (int)rintf(__fdiv_rn(v[e], s));
            q = max(-8, min(7, q));
        }
        const int nib = (e & 1) ? 4 + (e >> 1) : (e >> 1);
        word |= (uint32_t)(q + 8) << (4 * nib);
    }
    *reinterpret_cast<uint32_t*>(packed + (size_t)row * (k / 2) + k0 / 2) = word;
    if ((lane & 7) == 0) {
        const int grp = (kb * 256 + lane * 8) / 64;
        scales[(size_t)grp * n + row] = *reinterpret_cast<const uint16_t*>(&sb);
    }
}

// Self-test of the bounded wait: waits on an mbarrier that nothing arrives
// on; the wait gives up after limit_ns and records DERR_TIMEOUT.
__global__ void selftest_wait_kernel(DevState* st, unsigned long long limit_ns) {
    pdl_trigger();
    pdl_wait();
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait_bounded(&bar, 0, limit_ns)) set_error(st, DERR_TIMEOUT, 300);
}

// Progress words of the round state: finished, tokens generated, KV length,
// tokens emitted by rounds (low 32 bits).
__global__ void progress_kernel(const DevState* st, int32_t* out) {
    pdl_trigger();
    pdl_wait();
    if (threadIdx.x != 0) return;
    out[0] = st->finished;
    out[1] = st->generated;
    out[2] = st->n;
    out[3] = (int32_t)st->emitted;
}

inline int ok(cudaError_t e) { return e == cudaSuccess ? 0 : -1; }

}  // namespace

int launch_prepare_rows(const RowsArgs& a, cudaStream_t s) {
    return ok(launch_k(prepare_rows_kernel, dim3(DFL_MAX_ROWS), dim3(256), 0, s, a));
}

int launch_attention(const AttnArgs& a, cudaStream_t s) {
    const int threads = 256;
    const size_t smem =
        (size_t)(2 * ATTN_CHUNK * a.head_dim + (threads / 32) * (ATTN_CHUNK + a.head_dim)) * 4;
    const dim3 g1(a.n_kv, a.max_chunks);
    if (a.head_dim == 128) {
        static bool set = false;
        if (!set) {
            if (cudaFuncSetAttribute(attn_partial_kernel<128>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
                return -1;
            set = true;
        }
        if (ok(launch_k(attn_partial_kernel<128>, g1, dim3(threads), smem, s, a))) return -1;
    } else if (a.head_dim == 64) {
        static bool set = false;
        if (!set) {
            if (cudaFuncSetAttribute(attn_partial_kernel<64>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
                return -1;
            set = true;
        }
        if (ok(launch_k(attn_partial_kernel<64>, g1, dim3(threads), smem, s, a))) return -1;
    } else {
        return -2;
    }
    return launch_attention_combine(a, s);
}

int launch_attention_combine(const AttnArgs& a, cudaStream_t s) {
    const dim3 g2(a.n_q, DFL_MAX_ROWS);
    if (a.head_dim == 128) return ok(launch_k(attn_combine_kernel<128>, g2, dim3(128), 0, s, a));
    if (a.head_dim == 64) return ok(launch_k(attn_combine_kernel<64>, g2, dim3(64), 0, s, a));
    return -2;
}

int launch_accept(const AcceptArgs& a, cudaStream_t s) {
    return ok(launch_k(accept_kernel, dim3(1), dim3(32), 0, s, a));
}

int launch_set_chunk(DevState* st, int pos0, int T, int commit_lo, cudaStream_t s) {
    return ok(launch_k(set_chunk_kernel, dim3(1), dim3(1), 0, s, st, pos0, T, commit_lo));
}

int launch_rollback(DevState* st, int new_len, int token, int block_max, int max_seq,
                    cudaStream_t s) {
    return ok(launch_k(rollback_kernel, dim3(1), dim3(1), 0, s, st, new_len, token, block_max,
                       max_seq));
}

int launch_set_ext_state(DevState* st, int n_ext, int first_token, int max_new, int block_max,
                         int max_seq, int eos_id, cudaStream_t s) {
    return ok(launch_k(set_ext_state_kernel, dim3(1), dim3(1), 0, s, st, n_ext, first_token,
                       max_new, block_max, max_seq, eos_id));
}

int launch_tap_reduce(const TapArgs& a, cudaStream_t s) {
    const long long vecs = (long long)a.rows * a.n_layers * a.hidden / 8;
    const int threads = 256;
    long long blocks = (vecs + threads - 1) / threads;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    const dim3 g((unsigned)blocks), b(threads);
    if (a.in_type == XT_BF16 && a.out_type == XT_F32)
        return ok(launch_k(tap_reduce_kernel<__nv_bfloat16, float>, g, b, 0, s, a));
    if (a.in_type == XT_BF16 && a.out_type == XT_BF16)
        return ok(launch_k(tap_reduce_kernel<__nv_bfloat16, __nv_bfloat16>, g, b, 0, s, a));
    if (a.in_type == XT_BF16 && a.out_type == XT_BF16S) {
        if (a.rows > DFL_MAX_ROWS && !a.lo_offset) return -2;   // the lo plane sits 16 rows below
        return ok(launch_k(tap_reduce_kernel<__nv_bfloat16, __nv_bfloat16, true>, g, b, 0, s, a));
    }
    if (a.in_type == XT_F32 && a.out_type == XT_F32)
        return ok(launch_k(tap_reduce_kernel<float, float>, g, b, 0, s, a));
    return -2;
}

int launch_ctx_rows(const CtxRowsArgs& a, cudaStream_t s) {
    if (a.rows < 1) return 0;
    return ok(launch_k(ctx_rows_kernel, dim3((unsigned)a.rows), dim3(256), 0, s, a));
}

int launch_dequant_int4g64_f16(const uint8_t* packed, const uint16_t* scales, int n, int k, void* out,
                               cudaStream_t s) {
    const long long words = (long long)n * (k / 8);
    long long blocks = (words + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    return ok(launch_k(dequant_int4g64_f16_kernel, dim3((unsigned)blocks), dim3(256), 0, s,
                       reinterpret_cast<const uint32_t*>(packed), scales, n, k,
                       reinterpret_cast<__half*>(out)));
}

int launch_embed_rows(const int32_t* tokens, int rows, const void* embed, int hidden, int vocab, float* x,
                      DevState* st, cudaStream_t s) {
    if (rows < 1) return 0;
    return ok(launch_k(embed_rows_kernel, dim3((unsigned)rows), dim3(256), 0, s, tokens, rows,
                       reinterpret_cast<const __nv_bfloat16*>(embed), hidden, vocab, x, st));
}

int launch_resid_norm(const ResidNormArgs& a, cudaStream_t s) {
    if (a.rows < 1) return 0;
    if (a.rows > 512)
        return ok(launch_k(resid_norm_wide_kernel, dim3((unsigned)a.rows), dim3(RN_THREADS), 0, s, a));
    return ok(launch_k(resid_norm_kernel, dim3((unsigned)a.rows), dim3(RN_THREADS), 0, s, a));
}

int launch_qkv_rows(const QkvRowsArgs& a, cudaStream_t s) {
    if (a.rows < 1) return 0;
    const long long warps = (long long)a.rows * (a.n_q + 2 * a.n_kv);
    return ok(launch_k(qkv_rows_kernel, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, s, a));
}

int launch_rope_rows(int pos0, int rows, int half, const double* inv_freq, float* cos_out, float* sin_out,
                     cudaStream_t s) {
    if (rows < 1) return 0;
    long long blocks = ((long long)rows * half + 255) / 256;
    if (blocks > 152 * 8) blocks = 152 * 8;
    return ok(launch_k(rope_rows_kernel, dim3((unsigned)blocks), dim3(256), 0, s, pos0, rows, half, inv_freq,
                       cos_out, sin_out));
}

int launch_ctx_kv_store(const CtxKvArgs& a, cudaStream_t s) {
    if (a.rows < 1) return 0;
    const long long warps = (long long)a.rows * a.n_kv * 2;
    return ok(launch_k(ctx_kv_store_kernel, dim3((unsigned)((warps + 7) / 8)), dim3(256), 0, s, a));
}

int launch_progress(const DevState* st, int32_t* out, cudaStream_t s) {
    return ok(launch_k(progress_kernel, dim3(1), dim3(32), 0, s, st, out));
}

int launch_selftest_wait(DevState* st, unsigned long long limit_ns, cudaStream_t s) {
    return ok(launch_k(selftest_wait_kernel, dim3(1), dim3(32), 0, s, st, limit_ns));
}

int launch_quantize_int4g64(const float* w, int n, int k, uint8_t* packed, uint16_t* scales,
                            cudaStream_t s) {
    const long long warps = (long long)n * (k / 256);
    const int per_block = 8;
    return ok(launch_k(quantize_int4g64_kernel, dim3((unsigned)((warps + per_block - 1) / per_block)),
                       dim3(per_block * 32), 0, s, w, n, k, packed, scales));
}

}  // namespace dfl
