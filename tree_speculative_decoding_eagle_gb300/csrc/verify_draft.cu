// Stage 4 with draft distributions: speculative-sampling verification of a
// tree whose tokens were drawn from the draft's distribution q.
//
// [EAGLE-1] section "検証方法": a drafted token is accepted by the ratio of the
// target and draft probabilities, min(1, p(t)/q(t)); after a rejection the
// target distribution is replaced by the residual norm(max(0, p - q)) and a
// token is finally drawn from it, so the output follows the target exactly.
// Tree form: at node cur the children (node order, all drafted from q =
// softmax(draft row of cur / T)) are tested in turn against the current
// residual R = max(0, p - C q) with normaliser S (C = 0, S = 1 before any
// rejection; each rejection adds S to C and recomputes S over the vocab):
//   child x with token t is accepted iff u[x,0] * S * q(t) < R(t).
// With no child accepted (or at a leaf) the bonus token is drawn from R by
// inverse CDF with u[cur,1].  A residual that sums to 0 falls back to p.
//
// One thread-block cluster of CL <= 8 CTAs per sequence; CTA r owns a
// contiguous slice of the vocabulary.  Every pass over the rows (per node:
// the (max, sum) of p and q; per rejection: S; for the bonus: the slices'
// masses) reduces within each CTA and then across the cluster: each CTA
// stores its partial into slot r of every CTA's shared memory and a cluster
// barrier completes the round, after which every CTA combines the CL
// partials in rank order.  So every CTA holds bitwise the same statistics,
// takes the same decisions (control flow is uniform across the cluster, and
// every CTA passes the same barriers), and the rows, which stay in L2, are
// read by CL SMs instead of one.  The bonus is drawn by the CTA whose slice
// holds the inverse CDF's threshold.
#include "common.cuh"
#include "sm100.cuh"

namespace eagle {

using sm100::cluster_arrive_relaxed;
using sm100::cluster_arrive_release;
using sm100::cluster_ctarank;
using sm100::cluster_wait;
using sm100::mapa_shared;
using sm100::smem_u32;
using sm100::st_cluster_f4;

constexpr int kVDThreads = 256;
constexpr int kVDMaxCluster = 8;
constexpr int kBatch = 4;  // vectors per thread whose loads are in flight together

struct DraftVerifyArgs {
  const void *target, *draft;
  int64_t ld_t, ld_d;
  const int32_t *node_tok, *node_parent, *node_row;
  int B, n, D, k, V;
  int CL;  // CTAs per sequence (the cluster size)
  float inv_t;
  const float *u;
  int32_t *accept_len, *path_nodes, *out_tokens, *status;
};

// Block-wide sum (all threads get it).  s_red holds one float per warp.
__device__ __forceinline__ float block_sum(float v, float *s_red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  float t = lane < nw ? s_red[lane] : 0.f;
  return warp_sum(t);
}

// Block-wide (max, sum of exp relative to max) merge of per-thread pairs.
__device__ __forceinline__ void block_lse(float &m, float &s, float *s_red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_combine(m, s, m2, s2);
  }
  __syncthreads();
  if (lane == 0) {
    s_red[2 * warp] = m;
    s_red[2 * warp + 1] = s;
  }
  __syncthreads();
  m = lane < nw ? s_red[2 * lane] : -INFINITY;
  s = lane < nw ? s_red[2 * lane + 1] : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
    lse_combine(m, s, m2, s2);
  }
}

template <typename T>
__global__ void __launch_bounds__(kVDThreads) verify_draft_kernel(DraftVerifyArgs a) {
  using VT = VecTraits<T>;
  constexpr int VEC = VT::kElems;
  constexpr int NT = kVDThreads;
  extern __shared__ __align__(16) int s_nodes[];
  int *s_par = s_nodes, *s_tok = s_nodes + a.n;
  __shared__ float s_red[64];
  __shared__ int s_kids[64 + 1];  // children of the current node (node order), count last
  __shared__ int s_pick;
  // cluster rounds: slot r of round parity p holds CTA r's partial
  __shared__ __align__(16) float4 s_x[2][kVDMaxCluster];
  const int b = blockIdx.y, tid = threadIdx.x, lane = tid & 31;
  const int CL = a.CL;
  const int rank = CL > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const int n = a.n, V = a.V, nvec = V / VEC;
  // this CTA's slice of the vocabulary, in 16-byte vectors
  const int per_cta = (nvec + CL - 1) / CL;
  const int c0 = min(nvec, rank * per_cta), c1 = min(nvec, c0 + per_cta), nv = c1 - c0;
  const float L2E = kLog2e;
  const float sc = a.inv_t * L2E;  // logit -> base-2 exponent units

  // one round: the block-uniform partial v goes to slot `rank` of every
  // CTA; after the barrier s_x[parity][0..CL) holds every CTA's partial.
  // Two parities: a CTA writes round j+2's slot only after every CTA has
  // arrived for round j+1, i.e. after every CTA has read round j.
  int xround = 0;
  auto exchange = [&](float4 v) -> const float4 * {
    const int par = xround & 1;
    ++xround;
    if (CL == 1) {
      if (tid == 0) s_x[par][0] = v;
      __syncthreads();
      return s_x[par];
    }
    if (tid < CL) st_cluster_f4(mapa_shared(smem_u32(&s_x[par][rank]), static_cast<uint32_t>(tid)), v);
    cluster_arrive_release();
    cluster_wait();
    return s_x[par];
  };

  pdl_wait();
  for (int i = tid; i < n; i += NT) {
    s_par[i] = a.node_parent[static_cast<int64_t>(b) * n + i];
    s_tok[i] = a.node_tok[static_cast<int64_t>(b) * n + i];
  }
  __syncthreads();
  if (CL > 1) {  // every CTA of the cluster is running before any remote store
    cluster_arrive_relaxed();
    cluster_wait();
  }

  int cur = 0, acc = 0;
  bool bad = false;
  for (int depth = 0;; ++depth) {
    // children of cur in node order (warp 0, ballot compaction)
    if (tid < 32) {
      int cnt = 0;
      for (int base = 0; base < n; base += 32) {
        const int i = base + lane;
        const bool kid = i > 0 && i < n && s_par[i] == cur;
        const unsigned bal = __ballot_sync(0xffffffffu, kid);
        const int pos = cnt + __popc(bal & ((1u << lane) - 1u));
        if (kid && pos < 64) s_kids[pos] = i;
        cnt += __popc(bal);
      }
      if (lane == 0) s_kids[64] = min(cnt, 64);
    }
    __syncthreads();
    const int nk = s_kids[64];
    const T *prow = reinterpret_cast<const T *>(a.target) + (static_cast<int64_t>(b) * n + cur) * a.ld_t;
    const T *qrow = nullptr;
    if (nk > 0) {
      const int r = a.node_row[static_cast<int64_t>(b) * n + cur];
      if (r < 0 || r >= a.D * a.k || depth >= a.D) {  // a parent must have been expanded
        bad = true;
        break;
      }
      qrow = reinterpret_cast<const T *>(a.draft) + (static_cast<int64_t>(b) * a.D * a.k + r) * a.ld_d;
    }
    // (max, sum) of p and q over this CTA's slice, in base-2 units: y = x *
    // inv_t * log2(e); each thread's vectors of a batch are loaded before
    // any is used, so a pass costs one memory latency per batch
    float mp = -INFINITY, sp = 0.f, mq = -INFINITY, sq = 0.f;
    for (int base = 0; base < nv; base += kBatch * NT) {
      uint4 bp[kBatch], bq[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const int vi = base + k * NT + tid;
        if (vi < nv) {
          bp[k] = *reinterpret_cast<const uint4 *>(prow + static_cast<int64_t>(c0 + vi) * VEC);
          if (qrow) bq[k] = *reinterpret_cast<const uint4 *>(qrow + static_cast<int64_t>(c0 + vi) * VEC);
        }
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        if (base + k * NT + tid >= nv) continue;
        float x[VEC];
        VT::unpack(bp[k], x);
        float vm = x[0];
#pragma unroll
        for (int e = 1; e < VEC; ++e) vm = fmaxf(vm, x[e]);
        vm *= sc;
        if (vm > -INFINITY) {  // a vector of -inf logits adds nothing
          const float mn = fmaxf(mp, vm);
          float acc_s = 0.f;
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc_s += ex2_approx(fmaf(x[e], sc, -mn));
          sp = (mp == -INFINITY ? 0.f : sp * ex2_approx(mp - mn)) + acc_s;
          mp = mn;
        }
        if (qrow) {
          VT::unpack(bq[k], x);
          float wm = x[0];
#pragma unroll
          for (int e = 1; e < VEC; ++e) wm = fmaxf(wm, x[e]);
          wm *= sc;
          if (wm > -INFINITY) {
            const float mq2 = fmaxf(mq, wm);
            float acc_q = 0.f;
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc_q += ex2_approx(fmaf(x[e], sc, -mq2));
            sq = (mq == -INFINITY ? 0.f : sq * ex2_approx(mq - mq2)) + acc_q;
            mq = mq2;
          }
        }
      }
    }
    // lse_combine works in natural units: the CTA's pairs, then the
    // cluster's CL pairs in rank order
    {
      float pm_n = mp * kLn2, ps = sp, qm_n = mq * kLn2, qs = sq;
      block_lse(pm_n, ps, s_red);
      if (qrow) block_lse(qm_n, qs, s_red);
      const float4 *x = exchange(make_float4(pm_n, ps, qm_n, qs));
      float pm = -INFINITY, pss = 0.f, qm = -INFINITY, qss = 0.f;
      for (int r = 0; r < CL; ++r) {
        const float4 v = x[r];
        lse_combine(pm, pss, v.x, v.y);
        lse_combine(qm, qss, v.z, v.w);
      }
      mp = pm * L2E;
      sp = pss;
      mq = qm * L2E;
      sq = qss;
    }
    const float ip = 1.f / sp, iq = qrow ? 1.f / sq : 0.f;
    // residual R(v) = max(0, p(v) - C q(v)), normaliser S
    float C = 0.f, S = 1.f;
    int accepted = -1;
    for (int c = 0; c < nk; ++c) {
      const int x = s_kids[c];
      const int t = s_tok[x];
      if (t < 0 || t >= V) {
        bad = true;
        break;
      }
      const float pt = ex2_approx(fmaf(VT::load1(prow, t), sc, -mp)) * ip;
      const float qt = ex2_approx(fmaf(VT::load1(qrow, t), sc, -mq)) * iq;
      const float ux = a.u[(static_cast<int64_t>(b) * n + x) * 2];
      if (ux * S * qt < fmaxf(0.f, pt - C * qt)) {
        accepted = x;
        break;
      }
      C += S;
      float part = 0.f;
      for (int base = 0; base < nv; base += kBatch * NT) {
        uint4 bp[kBatch], bq[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          const int vi = base + k * NT + tid;
          if (vi < nv) {
            bp[k] = *reinterpret_cast<const uint4 *>(prow + static_cast<int64_t>(c0 + vi) * VEC);
            bq[k] = *reinterpret_cast<const uint4 *>(qrow + static_cast<int64_t>(c0 + vi) * VEC);
          }
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
          if (base + k * NT + tid >= nv) continue;
          float xp[VEC], xq[VEC];
          VT::unpack(bp[k], xp);
          VT::unpack(bq[k], xq);
#pragma unroll
          for (int e = 0; e < VEC; ++e)
            part += fmaxf(0.f, ex2_approx(fmaf(xp[e], sc, -mp)) * ip - C * ex2_approx(fmaf(xq[e], sc, -mq)) * iq);
        }
      }
      part = block_sum(part, s_red);
      const float4 *xs = exchange(make_float4(part, 0.f, 0.f, 0.f));
      S = 0.f;
      for (int r = 0; r < CL; ++r) S += xs[r].x;
      if (!(S > 0.f)) {  // nothing left: fall back to p
        C = 0.f;
        S = 1.f;
      }
    }
    if (bad) break;
    if (accepted >= 0) {
      if (rank == 0 && tid == 0) {
        a.path_nodes[static_cast<int64_t>(b) * (a.D + 1) + acc + 1] = accepted;
        a.out_tokens[static_cast<int64_t>(b) * (a.D + 1) + acc] = s_tok[accepted];
      }
      cur = accepted;
      ++acc;
      continue;
    }
    // bonus: inverse CDF of R.  Thread t of CTA r owns a contiguous range of
    // the slice; the CTAs' masses are exchanged, and the CTA whose range of
    // the cumulative mass holds u * total draws the token.
    const int per = (nv + NT - 1) / NT;
    const int v0 = c0 + min(nv, tid * per), v1 = c0 + min(nv, tid * per + per);
    float own = 0.f;
    const bool use_q = qrow && C > 0.f;
    for (int vb = v0; vb < v1; vb += kBatch) {
      uint4 bp[kBatch], bq[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        if (vb + k < v1) {
          bp[k] = *reinterpret_cast<const uint4 *>(prow + static_cast<int64_t>(vb + k) * VEC);
          if (use_q) bq[k] = *reinterpret_cast<const uint4 *>(qrow + static_cast<int64_t>(vb + k) * VEC);
        }
      }
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        if (vb + k >= v1) continue;
        float xp[VEC], xq[VEC];
        VT::unpack(bp[k], xp);
        if (use_q) VT::unpack(bq[k], xq);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
          const float p = ex2_approx(fmaf(xp[e], sc, -mp)) * ip;
          own += use_q ? fmaxf(0.f, p - C * ex2_approx(fmaf(xq[e], sc, -mq)) * iq) : p;
        }
      }
    }
    // exclusive block scan of `own`, and the CTA's mass
    float incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    __syncthreads();
    if (lane == 31) s_red[tid >> 5] = incl;
    if (tid == 0) s_pick = -1;
    __syncthreads();
    float wbase = 0.f, mine = 0.f;
    for (int w = 0; w < (NT >> 5); ++w) {
      const float ws = s_red[w];
      if (w < (tid >> 5)) wbase += ws;
      mine += ws;
    }
    const float *xm = reinterpret_cast<const float *>(exchange(make_float4(mine, 0.f, 0.f, 0.f)));
    // the drawing CTA: the first whose cumulative range holds the
    // threshold; past the rounded total, the last CTA with mass
    float total = 0.f;
    for (int r = 0; r < CL; ++r) total += xm[4 * r];
    const float thr = a.u[(static_cast<int64_t>(b) * n + cur) * 2 + 1] * total;
    int sel = -1, last = -1;
    float sel_base = 0.f, last_base = 0.f, run = 0.f;
    for (int r = 0; r < CL; ++r) {
      const float mr = xm[4 * r];
      if (mr > 0.f) {
        if (sel < 0 && thr < run + mr) {
          sel = r;
          sel_base = run;
        }
        last = r;
        last_base = run;
      }
      run += mr;
    }
    bool past_end = false;
    if (sel < 0) {
      sel = last;
      sel_base = last_base;
      past_end = true;
    }
    if (sel == rank) {
      const float tl = past_end ? mine : thr - sel_base;  // the threshold within this CTA
      const float before = wbase + incl - own;
      if (!past_end && own > 0.f && tl >= before && tl < before + own) {
        float rr = before;
        int pick = -1;
        for (int vi = v0; vi < v1 && pick < 0; ++vi) {
          float xp[VEC], xq[VEC];
          VT::unpack(*reinterpret_cast<const uint4 *>(prow + static_cast<int64_t>(vi) * VEC), xp);
          if (use_q) VT::unpack(*reinterpret_cast<const uint4 *>(qrow + static_cast<int64_t>(vi) * VEC), xq);
          for (int e = 0; e < VEC; ++e) {
            const float p = ex2_approx(fmaf(xp[e], sc, -mp)) * ip;
            const float r = use_q ? fmaxf(0.f, p - C * ex2_approx(fmaf(xq[e], sc, -mq)) * iq) : p;
            rr += r;
            if (r > 0.f && rr > tl) {
              pick = vi * VEC + e;
              break;
            }
          }
        }
        if (pick < 0) pick = v1 * VEC - 1;  // rounding at the range's end
        atomicMax(&s_pick, pick);
      }
      __syncthreads();
      int bonus = s_pick;
      if (bonus < 0) {
        // the threshold at or beyond the CTA's rounded mass: its last token with mass
        if (own > 0.f) atomicMax(&s_pick, v1 * VEC - 1);
        __syncthreads();
        bonus = s_pick;
      }
      if (tid == 0) {
        a.out_tokens[static_cast<int64_t>(b) * (a.D + 1) + acc] = bonus;
        if (bonus < 0) report(a.status, EAGLE_ERR_INVALID);
      }
    } else if (sel < 0 && rank == 0 && tid == 0) {  // no mass anywhere
      a.out_tokens[static_cast<int64_t>(b) * (a.D + 1) + acc] = -1;
      report(a.status, EAGLE_ERR_INVALID);
    }
    break;
  }
  if (rank == 0 && tid == 0) {
    const int64_t ob = static_cast<int64_t>(b) * (a.D + 1);
    a.accept_len[b] = acc;
    a.path_nodes[ob] = 0;
    for (int i = acc + 1; i <= a.D; ++i) a.path_nodes[ob + i] = -1;
    if (bad) a.out_tokens[ob + acc] = -1;
    for (int i = acc + 1; i <= a.D; ++i) a.out_tokens[ob + i] = -1;
    if (bad) report(a.status, EAGLE_ERR_INVALID);
  }
}

// Cluster size: about 512 vectors of a row per CTA, at most 8 CTAs.
static int verify_draft_cluster(int V, int vec) {
  const int nvec = V / vec;
  int cl = (nvec + 511) / 512;
  if (cl > kVDMaxCluster) cl = kVDMaxCluster;
  return cl < 1 ? 1 : cl;
}

cudaError_t launch_verify_draft(const void *target, const void *draft, int dtype, int64_t ld_t, int64_t ld_d,
                                const int32_t *node_tok, const int32_t *node_parent, const int32_t *node_row,
                                int B, int m, int D, int k, int V, float temperature, const float *uniforms,
                                int32_t *accept_len, int32_t *path_nodes, int32_t *out_tokens, int32_t *status,
                                cudaStream_t st) {
  DraftVerifyArgs a;
  a.target = target; a.draft = draft; a.ld_t = ld_t; a.ld_d = ld_d;
  a.node_tok = node_tok; a.node_parent = node_parent; a.node_row = node_row;
  a.B = B; a.n = m + 1; a.D = D; a.k = k; a.V = V;
  a.CL = verify_draft_cluster(V, dtype == EAGLE_BF16 ? 8 : 4);
  a.inv_t = 1.f / temperature;
  a.u = uniforms;
  a.accept_len = accept_len; a.path_nodes = path_nodes; a.out_tokens = out_tokens; a.status = status;
  const size_t smem = sizeof(int) * 2 * static_cast<size_t>(a.n);
  const dim3 grid(a.CL, B);
  if (dtype == EAGLE_BF16)
    return launch_chained_cluster(verify_draft_kernel<__nv_bfloat16>, grid, dim3(kVDThreads), smem, st,
                                  static_cast<unsigned>(a.CL), a);
  return launch_chained_cluster(verify_draft_kernel<float>, grid, dim3(kVDThreads), smem, st,
                                static_cast<unsigned>(a.CL), a);
}

}  // namespace eagle
