// Stage 4: the verification walk over the draft tree.
//
// [EAGLE-1] section "検証方法": every draft token is accepted or rejected by
// the ratio of target and draft distributions; after a rejection the rest of
// the branch is discarded and a token is resampled, so the output follows
// the target model exactly ([EAGLE-2]: lossless; temp=0 is greedy).
// Children are point-mass drafts, so child x (token t) is accepted with
// probability equal to t's residual target probability:
//   accept iff u[x,0] * (Z - sum_{s in S} e_s) < e_t,
// and the bonus token is drawn from the residual by inverse CDF with u[cur,1].
//
// Two kernels:
//  (a) verify_stats: one pass over all target rows in HBM.  Each warp owns a
//      2048-token chunk of a row and records (max, sum exp(y - max), argmax)
//      of y = x / T; these do not depend on the tree, so the pass can run
//      beside the draft stages.
//  (b) verify_walk: one CTA per sequence first loads, in one parallel round,
//      every node's parent, token, logit in its parent's row and uniforms,
//      and the sequence's chunk statistics; one warp then walks the tree
//      from shared memory and, for a bonus draw, re-reads one chunk.
#include "common.cuh"

namespace eagle {

constexpr int kChunk = 2048;  // tokens per statistics chunk (64 per lane)

struct alignas(16) ChunkStat {
  float m;  // max of y over the chunk
  float s;  // sum of exp(y - m) over the chunk (sampling mode)
  int a;    // lowest token attaining m (greedy mode)
  int pad;
};

struct VerifyArgs {
  const void *target;
  int64_t ld;
  const int32_t *node_tok, *node_parent;
  int B, m, n, D, V, nch, mode;
  int stage_stats;  // walk: the sequence's chunk statistics are copied to shared memory first
  float inv_t;
  const float *u;
  int32_t *accept_len, *path_nodes, *out_tokens, *status;
  ChunkStat *stats;
};

template <typename T, bool SAMPLE>
__global__ void __launch_bounds__(256) verify_stats_kernel(VerifyArgs a) {
  using VT = VecTraits<T>;
  constexpr int VEC = VT::kElems;
  constexpr int NVL = kChunk / VEC / 32;  // vectors per lane
  const int lane = threadIdx.x & 31;
  const int64_t total = static_cast<int64_t>(a.B) * a.n * a.nch;
  const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  pdl_wait();
  for (int64_t task = wid; task < total; task += nwarps) {
    const int64_t row = task / a.nch;
    const int c = static_cast<int>(task % a.nch);
    const T *p = reinterpret_cast<const T *>(a.target) + row * a.ld;
    const int t_begin = c * kChunk;
    const int nvec = (min(a.V, t_begin + kChunk) - t_begin) / VEC;
    uint4 buf[NVL];
#pragma unroll
    for (int i = 0; i < NVL; ++i) {
      const int v = lane + 32 * i;
      if (v < nvec) buf[i] = ld_stream16(p + t_begin + v * VEC);
    }
    ChunkStat st;
    st.pad = 0;
    if (SAMPLE) {
      // max of the raw logits (packed max; scaling by 1/T > 0 keeps order,
      // so the chunk max of x/T is max(x) / T exactly), then
      // sum exp(x/T - M) with 1/T folded into the exponent's FMA
      float bx = -INFINITY;
#pragma unroll
      for (int i = 0; i < NVL; ++i)
        if (lane + 32 * i < nvec) bx = fmaxf(bx, vec_max<T>(buf[i]));
      const float M = from_ordered_u32(__reduce_max_sync(0xffffffffu, ordered_u32(bx))) * a.inv_t;
      float s0 = 0.f, s1 = 0.f;
      if (M > -INFINITY) {
        const float sc = a.inv_t * kLog2e, nmL = -M * kLog2e;
#pragma unroll
        for (int i = 0; i < NVL; ++i) {
          if (lane + 32 * i < nvec) {
            float x[VEC];
            VT::unpack(buf[i], x);
#pragma unroll
            for (int e = 0; e < VEC; e += 2) {
              s0 += ex2_approx(fmaf(x[e], sc, nmL));
              s1 += ex2_approx(fmaf(x[e + 1], sc, nmL));
            }
          }
        }
      }
      st.m = M;
      st.s = warp_sum(s0 + s1);
      st.a = -1;
    } else {
      float best = -INFINITY;
      int arg = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < NVL; ++i) {
        const int v = lane + 32 * i;
        if (v < nvec) {
          float x[VEC];
          VT::unpack(buf[i], x);
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            if (x[e] > best) {  // strict: first occurrence within the lane
              best = x[e];
              arg = t_begin + v * VEC + e;
            }
          }
        }
      }
      const uint32_t om = __reduce_max_sync(0xffffffffu, ordered_u32(best));
      st.m = from_ordered_u32(om);
      const uint32_t cand = (ordered_u32(best) == om) ? static_cast<uint32_t>(arg) : 0xffffffffu;
      st.a = static_cast<int>(__reduce_min_sync(0xffffffffu, cand));
      st.s = 0.f;
    }
    if (lane == 0) a.stats[task] = st;
  }
  pdl_trigger();
}

// logit of token t in row `row`, scaled by 1/T
template <typename T>
__device__ __forceinline__ float logit_at(const VerifyArgs &a, int64_t row, int t) {
  return VecTraits<T>::load1(a.target, row * a.ld + t);
}

constexpr int kWalkThreads = 256;

// The walk.  Every state the walk can visit is loaded first, by all eight
// warps in one round: each node's parent and token, its logit in its
// parent's row and its two uniforms (sampling), and the sequence's chunk
// statistics (when they fit in shared memory).  Warp 0 then walks, reducing
// the current row's chunk statistics at each step; only the sampling bonus
// reads the target again (one chunk).
template <typename T>
__global__ void __launch_bounds__(kWalkThreads) verify_walk_kernel(VerifyArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int n = a.n;
  ChunkStat *s_cs = reinterpret_cast<ChunkStat *>(smem);  // [n][nch] when staged
  int *s_par = reinterpret_cast<int *>(smem + (a.stage_stats ? sizeof(ChunkStat) * n * a.nch : 0));
  int *s_tok = s_par + n;
  int *s_rej = s_tok + n;  // rejected tokens at the current node
  float *s_rej_e = reinterpret_cast<float *>(s_rej + n);  // and their exp terms
  float *s_x = s_rej_e + n;   // node i's logit in its parent's row (sampling)
  float *s_u = s_x + n;       // [n][2] node i's uniforms (sampling)
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t nb = static_cast<int64_t>(b) * n;
  const float sc = a.inv_t * kLog2e;  // logit -> base-2 exponent of exp(x / T), as the statistics pass
  const bool sample = a.mode == EAGLE_SAMPLE;
  pdl_wait();
  if (a.stage_stats) {
    const uint4 *src = reinterpret_cast<const uint4 *>(a.stats + nb * a.nch);
    uint4 *dst = reinterpret_cast<uint4 *>(s_cs);
    const int total = n * a.nch;
#pragma unroll 8
    for (int q = tid; q < total; q += kWalkThreads) dst[q] = src[q];
  }
  for (int i = tid; i < n; i += kWalkThreads) {
    const int par = a.node_parent[nb + i], tk = a.node_tok[nb + i];
    s_par[i] = par;
    s_tok[i] = tk;
    if (sample) {
      float x = 0.f;
      if (i > 0 && par >= 0 && par < n && tk >= 0 && tk < a.V) x = logit_at<T>(a, nb + par, tk);
      s_x[i] = x;
      s_u[2 * i] = a.u[(nb + i) * 2 + 0];
      s_u[2 * i + 1] = a.u[(nb + i) * 2 + 1];
    }
  }
  __syncthreads();
  if (warp != 0) return;

  int cur = 0, acc = 0, bonus = -1;
  if (lane == 0) a.path_nodes[static_cast<int64_t>(b) * (a.D + 1)] = 0;

  for (;;) {
    const int64_t row = nb + cur;
    const ChunkStat *cs = (a.stage_stats ? s_cs : a.stats + nb * a.nch) + static_cast<int64_t>(cur) * a.nch;
    // row maximum (and, greedy, the argmax) from the chunk statistics
    float bm = -INFINITY;
    int ba = 0x7fffffff;
    for (int c = lane; c < a.nch; c += 32) {
      const ChunkStat st = cs[c];
      if (st.m > bm) { bm = st.m; ba = st.a; }  // chunks ascend in token order
    }
    const uint32_t om = __reduce_max_sync(0xffffffffu, ordered_u32(bm));
    const float M = from_ordered_u32(om);
    const float mL = M * kLog2e;
    int next = -1;
    float Z = 0.f, rej_sum = 0.f;
    int n_rej = 0;
    if (!sample) {
      bonus = static_cast<int>(__reduce_min_sync(
          0xffffffffu, ordered_u32(bm) == om ? static_cast<uint32_t>(ba) : 0xffffffffu));
      // a row with no finite logit (all -inf, or NaN) has no argmax: the walk
      // stops here with bonus -1 and reports EAGLE_ERR_INVALID below
      if (bonus < 0 || bonus >= a.V) bonus = -1;
      for (int base = 0; bonus >= 0 && base < n && next < 0; base += 32) {
        const int i = base + lane;
        const bool hit = i < n && s_par[i] == cur && s_tok[i] == bonus;
        const unsigned bal = __ballot_sync(0xffffffffu, hit);
        if (bal) next = base + __ffs(bal) - 1;
      }
    } else {
      float z = 0.f;
      for (int c = lane; c < a.nch; c += 32) {
        const ChunkStat st = cs[c];
        if (st.m > -INFINITY) z += st.s * ex2_approx(fmaf(st.m, kLog2e, -mL));
      }
      Z = warp_sum(z);
      for (int base = 0; base < n && next < 0; base += 32) {
        // the children among nodes base..base+31, in node order: every child
        // before the accepted one was rejected, so child j sees the residual
        // mass Z - rej_sum - (sum of e over the earlier children here), and
        // the accepted child is the first whose test passes (one scan, no
        // serial loop)
        const int i = base + lane;
        const bool kid = i < n && s_par[i] == cur;
        int t_l = -1;
        float e_l = 0.f, u_l = 0.f;
        if (kid) {
          t_l = s_tok[i];
          if (t_l >= 0 && t_l < a.V) e_l = ex2_approx(fmaf(s_x[i], sc, -mL));
          else report(a.status, EAGLE_ERR_INVALID);
          u_l = s_u[2 * i];
        }
        float incl = e_l;  // e_l is 0 off the children
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        const float excl = incl - e_l;
        const unsigned kids = __ballot_sync(0xffffffffu, kid);
        const unsigned acc_b = __ballot_sync(0xffffffffu, kid && u_l * (Z - rej_sum - excl) < e_l);
        const int first = acc_b ? __ffs(acc_b) - 1 : 32;  // the accepted child's lane
        const unsigned before = first < 32 ? kids & ((1u << first) - 1u) : kids;  // rejected children
        if ((before >> lane) & 1u) {
          const int pos = n_rej + __popc(before & ((1u << lane) - 1u));
          s_rej[pos] = (t_l >= 0 && t_l < a.V) ? t_l : -1;
          s_rej_e[pos] = e_l;
        }
        n_rej += __popc(before);
        rej_sum += __shfl_sync(0xffffffffu, first < 32 ? excl : incl, first < 32 ? first : 31);
        if (first < 32) next = base + first;
      }
      __syncwarp();
    }
    if (next < 0 || acc >= a.D) {
      if (sample) {
        // ---- bonus: inverse CDF of the residual over the row -------------
        // Warp-parallel throughout (one lane walking a run of tokens or
        // chunks with data-dependent branches was the walk's slowest part).
        // Sums are fp32: this part's fp64 pipe is a small fraction of its
        // fp32 rate.  A chunk's mass drops its rejected tokens' terms.
        const float tgt = s_u[2 * cur + 1] * (Z - rej_sum);
        auto chunk_mass = [&](int c) {
          const ChunkStat st = cs[c];
          float w = st.m > -INFINITY ? st.s * ex2_approx(fmaf(st.m, kLog2e, -mL)) : 0.f;
          for (int q = 0; q < n_rej; ++q) {
            const int t = s_rej[q];
            w -= (t >= 0 && t / kChunk == c) ? s_rej_e[q] : 0.f;
          }
          return fmaxf(w, 0.f);
        };
        // the chunk: rounds of 32 chunks (lane l takes chunk 32r + l), a
        // running total carried between rounds; the first chunk whose
        // inclusive sum exceeds the target, else the last chunk with mass
        int chunk = -1, last_c = -1;
        float before = 0.f, last_before = 0.f, carry = 0.f;
        for (int r0 = 0; r0 < a.nch && chunk < 0; r0 += 32) {
          const int c = r0 + lane;
          const float w = c < a.nch ? chunk_mass(c) : 0.f;
          float incl = w;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
          }
          const unsigned hit = __ballot_sync(0xffffffffu, w > 0.f && carry + incl > tgt);
          const unsigned nz = __ballot_sync(0xffffffffu, w > 0.f);
          if (hit) {
            const int hl = __ffs(hit) - 1;
            chunk = r0 + hl;
            before = carry + __shfl_sync(0xffffffffu, incl - w, hl);
          } else if (nz) {
            const int hl = 31 - __clz(nz);
            last_c = r0 + hl;
            last_before = carry + __shfl_sync(0xffffffffu, incl - w, hl);
          }
          carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (chunk < 0) {
          chunk = last_c;
          before = last_before;
        }
        if (chunk < 0) {  // no residual mass anywhere: inputs outside the domain
          bonus = -1;
          break;
        }
        // the chunk's tokens: lane l owns 64 consecutive tokens; rejected
        // tokens are masked out
        constexpr int VEC = VecTraits<T>::kElems, NV = 64 / VEC;
        const int tb = chunk * kChunk + lane * 64;
        const int te = min(a.V, tb + 64);
        uint64_t rejm = 0;  // rejected tokens inside [tb, te)
        for (int q = 0; q < n_rej; ++q) {
          const int t = s_rej[q];
          rejm |= (t >= tb && t < te) ? 1ull << (t - tb) : 0ull;
        }
        uint4 v[NV];
        const T *rp = reinterpret_cast<const T *>(a.target) + row * a.ld;
#pragma unroll
        for (int q = 0; q < NV; ++q)
          v[q] = tb + q * VEC < te ? *reinterpret_cast<const uint4 *>(rp + tb + q * VEC) : make_uint4(0u, 0u, 0u, 0u);
        float lane_w = 0.f;
#pragma unroll
        for (int q = 0; q < NV; ++q) {
          float x[VEC];
          VecTraits<T>::unpack(v[q], x);
#pragma unroll
          for (int e = 0; e < VEC; ++e) {
            const bool use = tb + q * VEC + e < te && !((rejm >> (q * VEC + e)) & 1ull);
            lane_w += use ? ex2_approx(fmaf(x[e], sc, -mL)) : 0.f;
          }
        }
        float lincl = lane_w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float vv = __shfl_up_sync(0xffffffffu, lincl, o);
          if (lane >= o) lincl += vv;
        }
        unsigned hitb = __ballot_sync(0xffffffffu, lane_w > 0.f && before + lincl > tgt);
        const unsigned nzb = __ballot_sync(0xffffffffu, lane_w > 0.f);
        const bool past_end = hitb == 0;  // rounding: the last token with mass
        const int hl2 = !past_end ? __ffs(hitb) - 1 : (nzb ? 31 - __clz(nzb) : 0);
        // the owning lane's 64 tokens, two per lane, read again (L2), with
        // its rejected-token mask and the mass before them
        const uint64_t orej = __shfl_sync(0xffffffffu, rejm, hl2);
        const float obefore = before + __shfl_sync(0xffffffffu, lincl - lane_w, hl2);
        const int ob = chunk * kChunk + hl2 * 64, oe = min(a.V, ob + 64);
        const int t0 = ob + 2 * lane, t1 = t0 + 1;
        float w0 = 0.f, w1 = 0.f;
        if (t0 < oe && !((orej >> (2 * lane)) & 1ull)) w0 = ex2_approx(fmaf(VecTraits<T>::load1(a.target, row * a.ld + t0), sc, -mL));
        if (t1 < oe && !((orej >> (2 * lane + 1)) & 1ull)) w1 = ex2_approx(fmaf(VecTraits<T>::load1(a.target, row * a.ld + t1), sc, -mL));
        float pincl = w0 + w1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float vv = __shfl_up_sync(0xffffffffu, pincl, o);
          if (lane >= o) pincl += vv;
        }
        const float r0 = obefore + (pincl - w0 - w1) + w0, r1 = r0 + w1;
        const bool h0 = w0 > 0.f && r0 > tgt, h1 = w1 > 0.f && r1 > tgt;
        const unsigned ph = __ballot_sync(0xffffffffu, !past_end && (h0 || h1));
        const unsigned pz = __ballot_sync(0xffffffffu, w0 > 0.f || w1 > 0.f);
        int tok = -1;
        if (ph) {
          const int l = __ffs(ph) - 1;
          tok = __shfl_sync(0xffffffffu, h0 ? t0 : t1, l);
        } else if (pz) {
          const int l = 31 - __clz(pz);
          tok = __shfl_sync(0xffffffffu, w1 > 0.f ? t1 : t0, l);
        }
        bonus = tok;
      }
      break;
    }
    cur = next;
    ++acc;
    if (lane == 0) {
      a.path_nodes[static_cast<int64_t>(b) * (a.D + 1) + acc] = cur;
      a.out_tokens[static_cast<int64_t>(b) * (a.D + 1) + acc - 1] = s_tok[cur];
    }
  }
  if (lane == 0) {
    const int64_t ob = static_cast<int64_t>(b) * (a.D + 1);
    a.accept_len[b] = acc;
    a.out_tokens[ob + acc] = bonus;
    for (int q = acc + 1; q <= a.D; ++q) {
      a.path_nodes[ob + q] = -1;
      a.out_tokens[ob + q] = -1;
    }
    if (bonus < 0) report(a.status, EAGLE_ERR_INVALID);
  }
  pdl_trigger();
}

// ---- host side ---------------------------------------------------------------

int verify_chunks(int V) { return (V + kChunk - 1) / kChunk; }

size_t verify_workspace_bytes(int B, int m, int V) {
  return sizeof(ChunkStat) * static_cast<size_t>(B) * (m + 1) * verify_chunks(V);
}

template <typename T>
static cudaError_t launch_verify_t(const VerifyArgs &a, int num_sms, cudaStream_t st) {
  const int64_t tasks = static_cast<int64_t>(a.B) * a.n * a.nch;
  int64_t blocks = (tasks + 7) / 8;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaError_t e = a.mode == EAGLE_SAMPLE
                      ? launch_chained(verify_stats_kernel<T, true>, dim3(static_cast<int>(blocks)), dim3(256), 0,
                                       st, a)
                      : launch_chained(verify_stats_kernel<T, false>, dim3(static_cast<int>(blocks)), dim3(256), 0,
                                       st, a);
  if (e != cudaSuccess) return e;
  size_t smem = sizeof(int) * 7 * static_cast<size_t>(a.n);
  if (a.stage_stats) smem += sizeof(ChunkStat) * static_cast<size_t>(a.n) * a.nch;
  if (smem > 48 * 1024) {
    static std::atomic<unsigned long long> configured{0};  // raised once per device, to the maximum
    e = set_smem_limit_max_once(verify_walk_kernel<T>, configured);
    if (e != cudaSuccess) return e;
  }
  return launch_chained(verify_walk_kernel<T>, dim3(a.B), dim3(kWalkThreads), smem, st, a);
}

cudaError_t launch_verify(const void *target, int dtype, int64_t ld, const int32_t *node_tok,
                          const int32_t *node_parent, int B, int m, int D, int V, int mode,
                          float temperature, const float *u, int32_t *accept_len,
                          int32_t *path_nodes, int32_t *out_tokens, int32_t *status, void *ws,
                          int num_sms, cudaStream_t st) {
  VerifyArgs a;
  a.target = target; a.ld = ld;
  a.node_tok = node_tok; a.node_parent = node_parent;
  a.B = B; a.m = m; a.n = m + 1; a.D = D; a.V = V;
  a.nch = verify_chunks(V);
  // the walk copies the chunk statistics of its sequence to shared memory
  // when they fit beside its other arrays
  a.stage_stats = sizeof(ChunkStat) * static_cast<size_t>(a.n) * a.nch + sizeof(int) * 7 * static_cast<size_t>(a.n) <=
                  200 * 1024;
  a.mode = mode;
  a.inv_t = mode == EAGLE_SAMPLE ? 1.0f / temperature : 1.0f;
  a.u = u;
  a.accept_len = accept_len; a.path_nodes = path_nodes; a.out_tokens = out_tokens;
  a.status = status;
  a.stats = reinterpret_cast<ChunkStat *>(ws);
  return dtype == EAGLE_BF16 ? launch_verify_t<__nv_bfloat16>(a, num_sms, st)
                             : launch_verify_t<float>(a, num_sms, st);
}

}  // namespace eagle
