// Sampler ladder of the multilingual T3 as an op-level kernel: classifier-
// free-guidance combine -> repetition penalty -> temperature -> min_p ->
// top-p -> top-k -> draw in vocabulary order ("Chatterbox -> ggml Port:
// Development Journal", the multilingual port's sampling path; the penalty
// divides positive logits and multiplies negative ones, as the journal's fix
// table records).  One CTA per row, every quantity in double precision; each
// probability is computed once (kept in shared memory beside the keys when
// they fit), only the entries min_p keeps are sorted, and the sort compares
// order-preserving 64-bit integer keys: this part's FP64 pipe is narrow, so FP64
// work is kept to one exp per entry:
//   z_i = c_i + w (c_i - u_i); seen i: z_i / penalty (z_i > 0) or z_i * penalty;
//   z_i / T; p_i = exp(z_i - max z)
//   min_p: keep p_i >= min(min_p, 1) (the largest probability is 1 here)
//   the survivors sorted by (z desc, index asc) with a bitonic sort of their
//   indices in shared memory (each comparison reads the two values); top-p: the
//   shortest prefix whose renormalised mass reaches top_p;
//   top-k: the prefix entries whose value is >= the k-th (ties kept)
//   draw: the smallest vocabulary index whose cumulative kept mass exceeds u
//   times the kept total.
#include "sd_internal.cuh"

namespace sd {
namespace ladder_detail {

constexpr int kT = 1024, kW = kT / 32;

__device__ __forceinline__ bool before(unsigned long long ka, int ia, unsigned long long kb, int ib) {
    return ka > kb || (ka == kb && ia < ib);
}

// Order-preserving 64-bit key of a double (the two zeros share one key); 0 is below every key
// of a number, so it marks the entries a stage has cut.  Integer compares instead of FP64 ones
// (the FP64 pipe of this part is narrow).
__device__ __forceinline__ unsigned long long ord_d(double z) {
    if (z == 0.0) z = 0.0;
    const unsigned long long b = (unsigned long long)__double_as_longlong(z);
    return (b >> 63) ? ~b : (b | 0x8000000000000000ull);
}

__device__ __forceinline__ double from_ord(unsigned long long k) {
    return __longlong_as_double((long long)((k >> 63) ? (k & 0x7FFFFFFFFFFFFFFFull) : ~k));
}

__device__ double block_max_d(double v, double* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmax(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    double r = red[0];
    for (int w = 1; w < kW; ++w) r = fmax(r, red[w]);
    __syncthreads();
    return r;
}

__device__ int block_min_i(int v, int* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    int r = red[0];
    for (int w = 1; w < kW; ++w) r = min(r, red[w]);
    __syncthreads();
    return r;
}

__device__ int block_max_i(int v, int* red) { return -block_min_i(-v, red); }

// exclusive scan of one double per thread in thread order (fixed order); *total = the sum
// exclusive scan of one int per thread in thread order; *total = the sum
__device__ int block_excl_scan_i(int v, int* red, int* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
    }
    if (lane == 31) red[warp] = inc;
    __syncthreads();
    int before_w = 0, tot = 0;
    for (int w = 0; w < kW; ++w) {
        if (w == warp) before_w = tot;
        tot += red[w];
    }
    __syncthreads();
    *total = tot;
    return before_w + inc - v;
}

__device__ double block_excl_scan_d(double v, double* red, double* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    double inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
    }
    if (lane == 31) red[warp] = inc;
    __syncthreads();
    double before_w = 0.0, tot = 0.0;
    for (int w = 0; w < kW; ++w) {
        if (w == warp) before_w = tot;
        tot += red[w];
    }
    __syncthreads();
    *total = tot;
    return before_w + inc - v;
}

__global__ void __launch_bounds__(kT) k_sample_ladder(const float* zc, const float* zu, int V, int NP, int keep_p,
                                                      float w, float pen, float T, float min_p, float top_p,
                                                      int top_k, const uint8_t* seen, const float* u, int32_t* out) {
    extern __shared__ __align__(16) unsigned char lsm[];
    // [V] ladder logits in vocabulary order, then (after the maximum) their order-preserving keys
    double* zv = reinterpret_cast<double*>(lsm);
    unsigned long long* kv = reinterpret_cast<unsigned long long*>(lsm);
    double* pv = zv + V;                             // [V] exp(z - max) when keep_p (each computed once)
    int* idx = reinterpret_cast<int*>(zv + (keep_p ? 2 * V : V));  // [NP] vocabulary index at each sorted position
    uint8_t* flag = reinterpret_cast<uint8_t*>(idx + NP);           // [V] kept after every stage
    __shared__ double dred[kW];
    __shared__ int ired[kW];
    const int row = blockIdx.x, tid = threadIdx.x;
    const float* c = zc + (size_t)row * V;
    const float* un = zu ? zu + (size_t)row * V : nullptr;
    const uint8_t* sn = seen ? seen + (size_t)row * V : nullptr;

    // ---- combine, penalty
    for (int i = tid; i < V; i += kT) {
        double z = c[i];
        if (un && w != 0.0f) z = z + (double)w * (z - (double)un[i]);
        if (sn && pen != 1.0f && sn[i]) z = z > 0.0 ? z / (double)pen : z * (double)pen;
        zv[i] = z;
    }
    __syncthreads();
    if (T <= 0.0f) {  // argmax, lowest index on ties
        double best = -INFINITY;
        int bi = 0x7fffffff;
        for (int i = tid; i < V; i += kT)
            if (zv[i] > best) { best = zv[i]; bi = i; }
        const double mx = block_max_d(best, dred);
        const int tok = block_min_i(best == mx ? bi : 0x7fffffff, ired);
        if (tid == 0) out[row] = tok;
        return;
    }
    // ---- temperature, max
    double lm = -INFINITY;
    for (int i = tid; i < V; i += kT) {
        zv[i] /= (double)T;
        lm = fmax(lm, zv[i]);
    }
    const double m = block_max_d(lm, dred);  // its barrier also publishes zv
    const double mp = min_p < 1.0f ? (double)min_p : 1.0;
    // ---- probabilities and keys; min_p: the entries it cuts take key 0
    for (int j = tid; j < V; j += kT) {
        const double z = zv[j], p = exp(z - m);
        if (keep_p) pv[j] = p;
        kv[j] = (min_p > 0.0f && !(p >= mp)) ? 0ull : ord_d(z);
    }
    __syncthreads();
    // ---- the entries min_p keeps, compacted in vocabulary order; the sort runs over the next
    // power of two, the positions past them holding V (key 0: they sort last)
    int NPc = 1;
    {
        const int seg0 = (V + kT - 1) / kT, a0 = min(V, tid * seg0), a1 = min(V, a0 + seg0);
        int cnt = 0;
        for (int i = a0; i < a1; ++i) cnt += kv[i] != 0ull;
        int total;
        int off = block_excl_scan_i(cnt, ired, &total);
        for (int i = a0; i < a1; ++i)
            if (kv[i] != 0ull) idx[off++] = i;
        while (NPc < total) NPc <<= 1;
        for (int j = total + tid; j < NPc; j += kT) idx[j] = V;
    }
    __syncthreads();
    auto key = [&](int t) -> unsigned long long { return idx[t] < V ? kv[idx[t]] : 0ull; };
    // exp(z - m) of vocabulary entry i (a survivor)
    auto prob = [&](int i) -> double { return keep_p ? pv[i] : exp(from_ord(kv[i]) - m); };
    // ---- bitonic sort: (z desc, index asc)
    for (int k = 2; k <= NPc; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < NPc; i += kT) {
                const int l = i ^ j;
                if (l <= i) continue;
                const bool up = (i & k) == 0;  // this pair's block sorts in the "before" order
                const int ii = idx[i], il = idx[l];
                const unsigned long long ki = ii < V ? kv[ii] : 0ull, kl = il < V ? kv[il] : 0ull;
                const bool swap = up ? before(kl, il, ki, ii) : before(ki, ii, kl, il);
                if (swap) {
                    idx[i] = il;
                    idx[l] = ii;
                }
            }
            __syncthreads();
        }
    }
    // survivors: the prefix of live keys
    int ns = 0;
    {
        int last = -1;
        for (int t = tid; t < NPc; t += kT)
            if (key(t) != 0ull) last = max(last, t);
        ns = block_max_i(last, ired) + 1;
    }
    // ---- top-p over the survivors: contiguous segments per thread, prefix of masses
    const int seg = (NPc + kT - 1) / kT, t0 = min(NPc, tid * seg), t1 = min(NPc, t0 + seg);
    if (top_p < 1.0f) {
        double loc = 0.0;
        for (int t = t0; t < t1; ++t)
            if (t < ns) loc += prob(idx[t]);
        double mass;
        double run = block_excl_scan_d(loc, dred, &mass);
        int cut = 0x7fffffff;
        for (int t = t0; t < t1 && t < ns; ++t) {
            run += prob(idx[t]);
            if (run / mass >= (double)top_p) { cut = t; break; }
        }
        cut = block_min_i(cut, ired);
        if (cut < ns) ns = cut + 1;
    }
    // ---- top-k over those: the prefix entries whose value is >= the k-th
    if (top_k >= 1 && top_k < ns) {
        const unsigned long long thr = key(top_k - 1);
        int last = -1;
        for (int t = tid; t < ns; t += kT)
            if (key(t) >= thr) last = max(last, t);
        ns = block_max_i(last, ired) + 1;
    }
    // ---- kept flags in vocabulary order
    for (int i = tid; i < V; i += kT) flag[i] = 0;
    __syncthreads();
    for (int t = tid; t < ns; t += kT) flag[idx[t]] = 1;
    __syncthreads();
    // ---- draw in vocabulary order
    const int vseg = (V + kT - 1) / kT, v0 = min(V, tid * vseg), v1 = min(V, v0 + vseg);
    double loc = 0.0;
    for (int i = v0; i < v1; ++i)
        if (flag[i]) loc += prob(i);
    double zs;
    double run = block_excl_scan_d(loc, dred, &zs);
    const double target = (double)u[row] * zs;
    int cand = 0x7fffffff, lastk = -1;
    for (int i = v0; i < v1; ++i) {
        if (!flag[i]) continue;
        lastk = i;
        run += prob(i);
        if (run > target) { cand = i; break; }
    }
    int tok = block_min_i(cand, ired);
    const int lastv = block_max_i(lastk, ired);
    if (tok == 0x7fffffff) tok = lastv;  // u * total rounded onto the last edge
    if (tid == 0) out[row] = tok;
}

// The decode step's ladder (one token for a conditional / unconditional row
// pair): before it, the token this step consumed joins the history mask (the
// tokens fed forward since the prompt; none in the prompt's own step) and row
// 0's draw goes to the ladder's input slot; after it, the token goes to both
// rows and to the step's output sequence.
__global__ void k_ladder_prep(const float* u1, const float* const* u_seq, const int* step_idx, int rows, float* u,
                              const int* prompt_on, const int32_t* consumed, int V, uint8_t* seen) {
    if (threadIdx.x != 0) return;
    *u = *u_seq ? (*u_seq)[(size_t)(*step_idx) * rows] : u1[0];
    const int t = consumed[0];
    if (!*prompt_on && t >= 0 && t < V) seen[t] = 1;
}

__global__ void k_ladder_commit(const int32_t* t_in, int32_t* tok, int rows, int V, int32_t* const* out_seq,
                                const int* step_idx, int* err) {
    if (threadIdx.x != 0) return;
    int t = *t_in;
    if (t < 0 || t >= V) {
        atomicCAS(err, 0, 2);
        t = 0;
    }
    for (int b = 0; b < rows; ++b) {
        tok[b] = t;
        if (*out_seq) (*out_seq)[(size_t)(*step_idx) * rows + b] = t;
    }
}

}  // namespace ladder_detail

cudaError_t launch_ladder_step(const float* logits, int ld, int rows, int V, const LadderParams& p, uint8_t* seen,
                               const int* prompt_on, const int32_t* consumed, const float* u1,
                               const float* const* u_seq, const int* step_idx, float* u_slot, int32_t* t_slot,
                               int32_t* tok, int32_t* const* out_seq, int* err, cudaStream_t st) {
    using namespace ladder_detail;
    k_ladder_prep<<<1, 32, 0, st>>>(u1, u_seq, step_idx, rows, u_slot, prompt_on, consumed, V, seen);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = launch_sample_ladder(logits, logits + ld, 1, V, p, seen, u_slot, t_slot, st);
    if (e != cudaSuccess) return e;
    k_ladder_commit<<<1, 32, 0, st>>>(t_slot, tok, rows, V, out_seq, step_idx, err);
    return cudaGetLastError();
}

namespace {
constexpr size_t kLadderSmemMax = 227 * 1024;
size_t ladder_bytes(int V, bool keep_p) {
    int NP = 1;
    while (NP < V) NP <<= 1;
    return (size_t)V * 8 * (keep_p ? 2 : 1) + (size_t)NP * 4 + (((size_t)V + 15) & ~(size_t)15);
}
// the probabilities are kept (one exp per entry) when they fit beside the keys
bool ladder_keep_p(int V) { return ladder_bytes(V, true) <= kLadderSmemMax; }
}  // namespace

size_t sample_ladder_smem_bytes(int V) { return ladder_bytes(V, ladder_keep_p(V)); }

cudaError_t launch_sample_ladder(const float* zc, const float* zu, int rows, int V, const LadderParams& p,
                                 const uint8_t* seen, const float* u, int32_t* out, cudaStream_t st) {
    using namespace ladder_detail;
    int NP = 1;
    while (NP < V) NP <<= 1;
    const size_t smem = sample_ladder_smem_bytes(V);
    cudaError_t e = cudaFuncSetAttribute(k_sample_ladder, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_sample_ladder<<<rows, kT, smem, st>>>(zc, zu, V, NP, ladder_keep_p(V) ? 1 : 0, p.cfg_weight, p.rep_penalty,
                                            p.temperature, p.min_p, p.top_p, p.top_k, seen, u, out);
    return cudaGetLastError();
}

}  // namespace sd
