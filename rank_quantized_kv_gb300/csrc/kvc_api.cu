// Host side of libkvc: descriptor validation, store layout, the frozen
// parameter block in kernel layouts, and the kvc_* C entry points.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "kvc_internal.h"
#include "kvc_tc.h"

using kvc::Params;

constexpr uint64_t kDefaultWaitNs = 2000000000ull;

struct kvc_layer {
  Params p{};
  void* block = nullptr;  // device parameter block (owned)
  int device = 0;
  int64_t len = 0;
  int64_t capacity = 0;
  int32_t path = KVC_PATH_AUTO;
  uint64_t wait_ns = kDefaultWaitNs;  // limit of the kernels' loop waits
  int64_t launches = 0;              // kernels launched by this layer (host count)
  int mode = 0, B = 0, H = 0, D = 0, hpg = 1, r = 0, n_bases = 0, n_slots = 0;
  int side_bytes = 0;
  int ncpos = 0;                     // largest chunk-aligned packed positions of a basis
  int pmax = 0;                      // largest packed row
  int64_t fixed_bytes = 0;
  std::vector<int32_t> P_host;       // per basis
  std::vector<int32_t> basis_host;   // per slot
  std::vector<int64_t> pay_host, side_host;
  std::vector<int32_t> seg_host;     // [nb][kMaxSeg][4] width segments
  kvc::TcPlan tc{};                  // tensor-core path tables (kvc_tc.cu)
};

namespace {

thread_local std::string g_err;

kvc_status fail(kvc_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

kvc_status succeed() {
  g_err.clear();
  return KVC_OK;
}

kvc_status cuda_fail(cudaError_t e, const char* what) {
  return fail(KVC_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

bool valid_width(int b) { return b == 0 || b == 1 || b == 2 || b == 3 || b == 4 || b == 8; }

}  // namespace

namespace kvc {

// Store layout: per slot, payload rows then side words, 256-byte aligned, each
// region with 16 bytes of slack for vector over-reads.
static void layout_store(const kvc_layer_desc* d, Geo& g) {
  g.pay_off.assign(g.n_slots, 0);
  g.side_off.assign(g.n_slots, 0);
  int64_t cur = 0;
  for (int s = 0; s < g.n_slots; ++s) {
    const int64_t P = d->mode == KVC_MODE_INT8 ? d->D : g.P[g.basis[s]];
    cur = align_up(cur, 256);
    g.pay_off[s] = cur;
    cur += d->capacity * P + 16;
    cur = align_up(cur, 256);
    g.side_off[s] = cur;
    cur += d->capacity * g.side_bytes + 16;
  }
  g.store_total = align_up(cur, 256);
}

kvc_status build_geo(const kvc_layer_desc* d, Geo& g) {
  if (!d) return fail(KVC_EINVAL, "descriptor is NULL");
  if (d->mode < KVC_MODE_UNIFORM || d->mode > KVC_MODE_INT8)
    return fail(KVC_EINVAL, "mode %d is not a KVC_MODE_*", d->mode);
  if (d->B <= 0 || d->H <= 0 || d->D <= 0) return fail(KVC_EINVAL, "B, H, D must be > 0");
  if (d->heads_per_group <= 0 || d->H % d->heads_per_group)
    return fail(KVC_EINVAL, "heads_per_group must be >= 1 and divide H");
  if (d->heads_per_group != 1 && d->mode != KVC_MODE_GROUP)
    return fail(KVC_EINVAL, "heads_per_group != 1 needs KVC_MODE_GROUP");
  if (d->in_dtype != KVC_F32 && d->in_dtype != KVC_F16 && d->in_dtype != KVC_BF16)
    return fail(KVC_EINVAL, "in_dtype must be KVC_F32, KVC_F16 or KVC_BF16");
  if (d->out_dtype != KVC_F16 && d->out_dtype != KVC_BF16)
    return fail(KVC_EINVAL, "out_dtype must be KVC_F16 or KVC_BF16");
  if (d->capacity < 1) return fail(KVC_EINVAL, "capacity must be >= 1");
  g.Hg = d->H / d->heads_per_group;
  g.d_in = d->heads_per_group * d->D;
  g.n_slots = d->B * g.Hg;
  if ((int64_t)d->B * g.Hg > (1 << 30)) return fail(KVC_EINVAL, "too many slots");

  if (d->mode == KVC_MODE_INT8) {
    g.nb = 0;
    g.r = 0;
    g.side_bytes = 2;
    g.basis.assign(g.n_slots, 0);
    g.P.assign(1, d->D);
  } else {
    if (d->r < 1 || d->r > kvc::kMaxRank || d->r > g.d_in)
      return fail(KVC_EINVAL, "r must be in [1, min(D_in, %d)]", kvc::kMaxRank);
    if (d->n_bases < 1) return fail(KVC_EINVAL, "n_bases must be >= 1");
    if (!d->V) return fail(KVC_EINVAL, "V is NULL");
    g.r = d->r;
    g.nb = d->n_bases;
    g.basis.assign(g.n_slots, 0);
    if (d->basis_of) {
      for (int s = 0; s < g.n_slots; ++s) {
        if (d->basis_of[s] < 0 || d->basis_of[s] >= g.nb)
          return fail(KVC_EINVAL, "basis_of[%d] = %d outside [0, %d)", s, d->basis_of[s], g.nb);
        g.basis[s] = d->basis_of[s];
      }
    }
    g.bits.assign((size_t)g.nb * g.r, 0);
    if (d->mode == KVC_MODE_CODEBOOK) {
      if (d->r != g.d_in) return fail(KVC_EINVAL, "codebook mode needs r == D");
      if (d->mean) return fail(KVC_EINVAL, "codebook mode takes no mean");
      const int cb = d->cb_bits;
      if (!(cb == 1 || cb == 2 || cb == 3 || cb == 4 || cb == 8))
        return fail(KVC_EINVAL, "cb_bits must be 1, 2, 3, 4 or 8");
      if (!d->codebook) return fail(KVC_EINVAL, "codebook is NULL");
      g.cb_levels = 1 << cb;
      for (int j = 0; j < g.cb_levels; ++j) {
        if (!std::isfinite(d->codebook[j])) return fail(KVC_EINVAL, "codebook has a non-finite entry");
        if (j && !(d->codebook[j] > d->codebook[j - 1]))
          return fail(KVC_EINVAL, "codebook must be strictly ascending");
      }
      std::fill(g.bits.begin(), g.bits.end(), (uint8_t)cb);
      g.side_bytes = 2;
    } else {
      if (!d->bits) return fail(KVC_EINVAL, "bits is NULL");
      for (size_t i = 0; i < g.bits.size(); ++i) {
        if (!valid_width(d->bits[i]))
          return fail(KVC_EINVAL, "bits[%zu] = %d is not in {0,1,2,3,4,8}", i, (int)d->bits[i]);
        g.bits[i] = d->bits[i];
      }
    }
    if (d->mode == KVC_MODE_UNIFORM) {
      if (!d->qmin || !d->qstep) return fail(KVC_EINVAL, "uniform mode needs qmin and qstep");
      for (size_t i = 0; i < g.bits.size(); ++i) {
        if (!g.bits[i]) continue;
        if (!std::isfinite(d->qmin[i]) || !std::isfinite(d->qstep[i]) || !(d->qstep[i] > 0.f))
          return fail(KVC_EINVAL, "qmin/qstep[%zu] must be finite with qstep > 0", i);
      }
    }
    if (d->mode == KVC_MODE_GROUP) {
      if (d->group_size < 1 || d->group_size > kvc::kMaxGroupSize)
        return fail(KVC_EINVAL, "group_size must be in [1, %d]", kvc::kMaxGroupSize);
      for (int b = 0; b < g.nb; ++b)
        for (int k = 0; k < g.r; ++k) {
          const int w = g.bits[(size_t)b * g.r + k];
          if (w == 1) return fail(KVC_EINVAL, "group mode needs widths >= 2 (or 0)");
          if (k && w > g.bits[(size_t)b * g.r + k - 1])
            return fail(KVC_EINVAL, "group mode needs non-increasing widths");
          if (w != g.bits[k]) return fail(KVC_EINVAL, "group mode needs the same widths for every basis");
        }
    }
    for (size_t i = 0; i < (size_t)g.nb * g.d_in * g.r; ++i)
      if (!std::isfinite(d->V[i])) return fail(KVC_EINVAL, "V has a non-finite entry");
    if (d->mean)
      for (size_t i = 0; i < (size_t)g.nb * g.d_in; ++i)
        if (!std::isfinite(d->mean[i])) return fail(KVC_EINVAL, "mean has a non-finite entry");

    // packed order and segments: widths descending, components ascending within a width
    g.P.assign(g.nb, 0);
    g.n_kept.assign(g.nb, 0);
    g.seg.assign((size_t)g.nb * kvc::kMaxSeg * 4, 0);
    g.order.assign((size_t)g.nb * g.r, (int16_t)-1);
    static const int kWidths[kvc::kMaxSeg] = {8, 4, 3, 2, 1};
    for (int b = 0; b < g.nb; ++b) {
      int m = 0, byte = 0, s = 0;
      for (int wi = 0; wi < kvc::kMaxSeg; ++wi) {
        const int w = kWidths[wi];
        int cnt = 0;
        for (int k = 0; k < g.r; ++k)
          if (g.bits[(size_t)b * g.r + k] == w) g.order[(size_t)b * g.r + m + cnt++] = (int16_t)k;
        if (!cnt) continue;
        int32_t* e = &g.seg[((size_t)b * kvc::kMaxSeg + s) * 4];
        e[0] = byte;
        e[1] = w;
        e[2] = m;
        e[3] = cnt;
        ++s;
        m += cnt;
        byte += (cnt * w + 7) / 8;
      }
      g.P[b] = byte;
      g.n_kept[b] = m;
    }
    if (d->mode == KVC_MODE_GROUP) {
      for (int s = 0; s < kvc::kMaxSeg; ++s) {
        const int32_t* e = &g.seg[(size_t)s * 4];
        if (!e[3]) break;
        const int first = g.order[e[2]];
        for (int o = 0; o < e[3]; o += d->group_size) {
          g.groups.push_back(first + o);
          g.groups.push_back(std::min(d->group_size, e[3] - o));
          g.groups.push_back(e[1]);
        }
      }
      g.n_groups = (int)g.groups.size() / 3;
      g.side_bytes = 2 * g.n_groups;
    }
  }

  layout_store(d, g);

  const int64_t din = g.d_in, r = g.r, nb = g.nb;
  // frozen parameters counted beside the codes: the basis and mean (fp32) of
  // every basis; uniform mode adds a width byte per component and an fp32
  // minimum and step per kept component; codebook and int8 modes count none
  switch (d->mode) {
    case KVC_MODE_UNIFORM: {
      int64_t kept = 0;
      for (int b = 0; b < g.nb; ++b) kept += g.n_kept[b];
      g.fixed = nb * (4 * din * r + 4 * din + r) + 8 * kept;
      break;
    }
    case KVC_MODE_GROUP: g.fixed = nb * (4 * din * r + 4 * din); break;
    default: g.fixed = 0;
  }
  return KVC_OK;
}

// A codebook key layer with a residual sketch and/or an outlier stream: the
// codebook geometry, then rows [indices | sign bytes | outlier codes] and side
// words [norm, residual norm, outlier scale].
kvc_status build_geo_prod(const kvc_layer_desc* d, const kvc_prod_desc* pd, Geo& g) {
  kvc_status st = build_geo(d, g);
  if (st) return st;
  if (!pd) return fail(KVC_EINVAL, "prod descriptor is NULL");
  if (d->mode != KVC_MODE_CODEBOOK) return fail(KVC_EINVAL, "the residual sketch needs KVC_MODE_CODEBOOK");
  if (g.nb != 1) return fail(KVC_EINVAL, "the residual sketch needs n_bases == 1");
  if (d->D != 32 && d->D != 64 && d->D != 128) return fail(KVC_EINVAL, "the residual sketch needs D in {32, 64, 128}");
  if (pd->m < 0 || pd->m > kProdMaxM || pd->m % 16)
    return fail(KVC_EINVAL, "m must be a multiple of 16 in [0, %d]", kProdMaxM);
  if (pd->m && !pd->S) return fail(KVC_EINVAL, "S is NULL");
  if (pd->n_outliers < 0 || pd->n_outliers > kProdMaxOut || pd->n_outliers >= d->D)
    return fail(KVC_EINVAL, "n_outliers must be in [0, min(%d, D - 1)]", kProdMaxOut);
  if (pd->n_outliers && !pd->channels) return fail(KVC_EINVAL, "channels is NULL");
  if (pd->split_from < 0) return fail(KVC_EINVAL, "split_from must be >= 0");
  g.S.assign((size_t)pd->m * d->D, 0.f);
  for (size_t i = 0; i < g.S.size(); ++i) {
    if (!std::isfinite(pd->S[i])) return fail(KVC_EINVAL, "S has a non-finite entry");
    g.S[i] = pd->S[i];
  }
  g.channels.assign((size_t)g.n_slots * pd->n_outliers, 0);
  for (int s = 0; s < g.n_slots; ++s)
    for (int l = 0; l < pd->n_outliers; ++l) {
      const int32_t c = pd->channels[(size_t)s * pd->n_outliers + l];
      if (c < 0 || c >= d->D || (l && c <= pd->channels[(size_t)s * pd->n_outliers + l - 1]))
        return fail(KVC_EINVAL, "channels of slot %d must be ascending and distinct in [0, D)", s);
      g.channels[(size_t)s * pd->n_outliers + l] = c;
    }
  g.prod = 1;
  g.m = pd->m;
  g.n_out = pd->n_outliers;
  g.split_from = pd->split_from;
  g.code_bytes = g.P[0];
  g.sign_bytes = (pd->m + 7) / 8;
  g.P[0] = g.code_bytes + g.sign_bytes + g.n_out;
  g.side_bytes = 2 * (1 + (g.m > 0) + (g.n_out > 0));
  layout_store(d, g);
  g.fixed = 0;
  return KVC_OK;
}

// The frozen parameters in kernel layouts (host image of the parameter block).
void build_param_image(const kvc_layer_desc* d, const Geo& g, ParamImage& im) {
  const int nb = g.nb, r = g.r, din = g.d_in;
  const bool coded = d->mode != KVC_MODE_INT8;
  std::vector<float> V, Vt, mean, lo, step, inv, vnorm, cb, mids;
  if (coded) {
    V.assign(d->V, d->V + (size_t)nb * din * r);
    Vt.assign((size_t)nb * r * din, 0.f);
    vnorm.assign((size_t)nb * r, 0.f);
    for (int b = 0; b < nb; ++b)
      for (int k = 0; k < r; ++k) {
        double ss = 0.0;
        for (int i = 0; i < din; ++i) {
          const float v = V[((size_t)b * din + i) * r + k];
          Vt[((size_t)b * r + k) * din + i] = v;
          ss += (double)v * v;
        }
        vnorm[(size_t)b * r + k] = std::nextafter((float)std::sqrt(ss), INFINITY);
      }
    mean.assign((size_t)nb * din, 0.f);
    if (d->mean) std::copy(d->mean, d->mean + (size_t)nb * din, mean.begin());
    lo.assign((size_t)nb * r, 0.f);
    step.assign((size_t)nb * r, 0.f);
    inv.assign((size_t)nb * r, 0.f);
    if (d->mode == KVC_MODE_UNIFORM)
      for (size_t i = 0; i < lo.size(); ++i) {
        if (!g.bits[i]) continue;
        lo[i] = d->qmin[i];
        step[i] = d->qstep[i];
        inv[i] = (float)(1.0 / (double)d->qstep[i]);
      }
    if (d->mode == KVC_MODE_CODEBOOK) {
      cb.assign(d->codebook, d->codebook + g.cb_levels);
      for (int j = 0; j + 1 < g.cb_levels; ++j)
        mids.push_back((float)(0.5 * ((double)cb[j] + (double)cb[j + 1])));
    }
  }

  im.oV = im.put(V.data(), V.size());
  im.oVt = im.put(Vt.data(), Vt.size());
  im.oMean = im.put(mean.data(), mean.size());
  im.oLo = im.put(lo.data(), lo.size());
  im.oStep = im.put(step.data(), step.size());
  im.oInv = im.put(inv.data(), inv.size());
  im.oVn = im.put(vnorm.data(), vnorm.size());
  im.oBits = im.put(g.bits.data(), g.bits.size());
  im.oOrder = im.put(g.order.data(), g.order.size());
  im.oSeg = im.put(g.seg.data(), g.seg.size());
  im.oP = im.put(g.P.data(), g.P.size());
  im.oKept = im.put(g.n_kept.data(), g.n_kept.size());
  im.oGroups = im.put(g.groups.data(), g.groups.size());
  im.oCb = im.put(cb.data(), cb.size());
  im.oMids = im.put(mids.data(), mids.size());
  im.oBasis = im.put(g.basis.data(), g.basis.size());
  im.oPay = im.put(g.pay_off.data(), g.pay_off.size());
  im.oSide = im.put(g.side_off.data(), g.side_off.size());
  im.oErr = im.zeros(sizeof(int));
  im.oCnt = im.zeros(4 * sizeof(unsigned long long));
  if (g.prod) {
    // W1 = [R | 0 | S^T from column 128], (S R)^T, W3 = [R^T ; S], row norms
    // rounded up; S R is formed in float64 and rounded once
    const int D = d->D, m = g.m;
    const float* R = d->V;
    std::vector<float> W1((size_t)D * 256, 0.f), SRt((size_t)D * 128, 0.f),
        W3((size_t)(D + m) * D, 0.f), sn(std::max(m, 1), 0.f), srn(std::max(m, 1), 0.f);
    for (int i = 0; i < D; ++i)
      for (int k = 0; k < D; ++k) {
        W1[(size_t)i * 256 + k] = R[(size_t)i * D + k];
        W3[(size_t)k * D + i] = R[(size_t)i * D + k];
      }
    for (int j = 0; j < m; ++j) {
      double s2 = 0.0, sr2 = 0.0;
      for (int i = 0; i < D; ++i) {
        const float v = g.S[(size_t)j * D + i];
        W1[(size_t)i * 256 + 128 + j] = v;
        W3[(size_t)(D + j) * D + i] = v;
        s2 += (double)v * v;
      }
      for (int k = 0; k < D; ++k) {
        double acc = 0.0;
        for (int i = 0; i < D; ++i) acc += (double)g.S[(size_t)j * D + i] * (double)R[(size_t)i * D + k];
        const float f = (float)acc;
        SRt[(size_t)k * 128 + j] = f;
        sr2 += (double)f * f;
      }
      sn[j] = std::nextafter((float)(std::sqrt(s2) * (1.0 + 1e-12)), INFINITY);
      srn[j] = std::nextafter((float)(std::sqrt(sr2) * (1.0 + 1e-12)), INFINITY);
    }
    im.oW1 = im.put(W1.data(), W1.size());
    im.oSRt = im.put(SRt.data(), SRt.size());
    im.oW3 = im.put(W3.data(), W3.size());
    im.oSn = im.put(sn.data(), sn.size());
    im.oSRn = im.put(srn.data(), srn.size());
    im.oCh = im.put(g.channels.data(), g.channels.size());
  }
}

// Device pointers of a parameter block uploaded from `im` at `base`.
void bind_params(Params& p, const kvc_layer_desc* d, const Geo& g, const ParamImage& im,
                 uint8_t* base) {
  p.mode = d->mode;
  p.B = d->B;
  p.H = d->H;
  p.D = d->D;
  p.hpg = d->heads_per_group;
  p.Hg = g.Hg;
  p.d_in = g.d_in;
  p.r = g.r;
  p.n_bases = g.nb;
  p.n_slots = g.n_slots;
  p.in_dtype = d->in_dtype;
  p.out_dtype = d->out_dtype;
  p.group_size = d->group_size;
  p.n_groups = g.n_groups;
  p.cb_levels = g.cb_levels;
  p.cb_bits = d->cb_bits;
  p.side_bytes = g.side_bytes;
  p.V = reinterpret_cast<const float*>(base + im.oV);
  p.Vt = reinterpret_cast<const float*>(base + im.oVt);
  p.mean = reinterpret_cast<const float*>(base + im.oMean);
  p.lo = reinterpret_cast<const float*>(base + im.oLo);
  p.step = reinterpret_cast<const float*>(base + im.oStep);
  p.inv_step = reinterpret_cast<const float*>(base + im.oInv);
  p.vnorm = reinterpret_cast<const float*>(base + im.oVn);
  p.bits = base + im.oBits;
  p.order = reinterpret_cast<const int16_t*>(base + im.oOrder);
  p.seg = reinterpret_cast<const int32_t*>(base + im.oSeg);
  p.P = reinterpret_cast<const int32_t*>(base + im.oP);
  p.n_kept = reinterpret_cast<const int32_t*>(base + im.oKept);
  p.groups = reinterpret_cast<const int32_t*>(base + im.oGroups);
  p.codebook = reinterpret_cast<const float*>(base + im.oCb);
  p.mids = reinterpret_cast<const float*>(base + im.oMids);
  p.basis_of = reinterpret_cast<const int32_t*>(base + im.oBasis);
  p.store = static_cast<uint8_t*>(d->store);
  p.pay_off = reinterpret_cast<const int64_t*>(base + im.oPay);
  p.side_off = reinterpret_cast<const int64_t*>(base + im.oSide);
  p.err = reinterpret_cast<int*>(base + im.oErr);
  p.counters = reinterpret_cast<unsigned long long*>(base + im.oCnt);
  if (g.prod) {
    p.prod = 1;
    p.m = g.m;
    p.n_out = g.n_out;
    p.code_bytes = g.code_bytes;
    p.sign_bytes = g.sign_bytes;
    p.split_from = g.split_from;
    p.W1 = reinterpret_cast<const float*>(base + im.oW1);
    p.SRt = reinterpret_cast<const float*>(base + im.oSRt);
    p.W3 = reinterpret_cast<const float*>(base + im.oW3);
    p.s_norm = reinterpret_cast<const float*>(base + im.oSn);
    p.sr_norm = reinterpret_cast<const float*>(base + im.oSRn);
    p.channels = reinterpret_cast<const int32_t*>(base + im.oCh);
  }
}

kvc_status set_error(kvc_status s, const char* msg) { return fail(s, "%s", msg); }

}  // namespace kvc

namespace {

using kvc::Geo;
using kvc::ParamImage;

bool is_device_ptr(const void* ptr, int dev) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, ptr) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) && at.device == dev;
}

struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

}  // namespace

namespace kvc {
bool device_ptr_on(const void* ptr, int dev) { return is_device_ptr(ptr, dev); }
}  // namespace kvc

extern "C" {

int32_t kvc_abi_version(void) { return KVC_ABI_VERSION; }

const char* kvc_last_error(void) { return g_err.c_str(); }

kvc_status kvc_store_bytes(const kvc_layer_desc* desc, size_t* out) {
  if (!out) return fail(KVC_EINVAL, "out is NULL");
  Geo g;
  kvc_status st = kvc::build_geo(desc, g);
  if (st) return st;
  *out = (size_t)g.store_total;
  return succeed();
}

static kvc_status init_from_geo(const kvc_layer_desc* d, Geo& g, kvc_layer** out);

kvc_status kvc_init_layer(const kvc_layer_desc* d, kvc_layer** out) {
  if (!out) return fail(KVC_EINVAL, "out is NULL");
  *out = nullptr;
  Geo g;
  kvc_status st = kvc::build_geo(d, g);
  if (st) return st;
  return init_from_geo(d, g, out);
}

kvc_status kvc_store_bytes_prod(const kvc_layer_desc* desc, const kvc_prod_desc* prod, size_t* out) {
  if (!out) return fail(KVC_EINVAL, "out is NULL");
  Geo g;
  kvc_status st = kvc::build_geo_prod(desc, prod, g);
  if (st) return st;
  *out = (size_t)g.store_total;
  return succeed();
}

kvc_status kvc_init_layer_prod(const kvc_layer_desc* d, const kvc_prod_desc* prod, kvc_layer** out) {
  if (!out) return fail(KVC_EINVAL, "out is NULL");
  *out = nullptr;
  Geo g;
  kvc_status st = kvc::build_geo_prod(d, prod, g);
  if (st) return st;
  return init_from_geo(d, g, out);
}

static kvc_status init_from_geo(const kvc_layer_desc* d, Geo& g, kvc_layer** out) {
  kvc_status st;
  if (!d->store) return fail(KVC_EINVAL, "store is NULL");
  if ((uintptr_t)d->store % 256) return fail(KVC_EINVAL, "store must be 256-byte aligned");
  if (d->store_bytes < (size_t)g.store_total)
    return fail(KVC_EINVAL, "store_bytes %zu < required %lld", d->store_bytes,
                (long long)g.store_total);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (!is_device_ptr(d->store, dev)) return fail(KVC_EINVAL, "store is not device memory of the current device");

  const int nb = g.nb, r = g.r, din = g.d_in;
  ParamImage im;
  kvc::build_param_image(d, g, im);

  kvc_layer* L = new kvc_layer();
  L->tc = kvc::TcPlan{};
  st = g.prod ? KVC_OK : kvc::tc_prepare(*d, g, im.bytes, L->tc);
  if (st) {
    delete L;
    return st;
  }

  void* block = nullptr;
  e = cudaMalloc(&block, im.bytes.size());
  if (e != cudaSuccess) {
    delete L;
    return cuda_fail(e, "cudaMalloc(parameter block)");
  }
  e = cudaMemcpy(block, im.bytes.data(), im.bytes.size(), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(block);
    delete L;
    return cuda_fail(e, "cudaMemcpy(parameter block)");
  }
  auto* base = static_cast<uint8_t*>(block);
  kvc::bind_params(L->p, d, g, im, base);
  kvc::tc_bind(L->tc, base);
  st = kvc::tc_alloc(L->tc, g.n_slots, r);
  if (st) {
    cudaFree(block);
    delete L;
    return st;
  }

  L->block = block;
  L->device = dev;
  L->capacity = d->capacity;
  L->mode = d->mode;
  L->B = d->B;
  L->H = d->H;
  L->D = d->D;
  L->hpg = d->heads_per_group;
  L->r = r;
  L->n_bases = nb;
  L->n_slots = g.n_slots;
  L->side_bytes = g.side_bytes;
  for (int b = 0; b < nb; ++b) {
    int pos = 0;
    for (int sg = 0; sg < kvc::kMaxSeg; ++sg) pos += (g.seg[((size_t)b * kvc::kMaxSeg + sg) * 4 + 3] + 7) / 8 * 8;
    L->ncpos = std::max(L->ncpos, pos);
    L->pmax = std::max(L->pmax, g.P[b]);
  }
  if (d->mode == KVC_MODE_INT8) L->pmax = d->D;
  L->fixed_bytes = g.fixed;
  L->P_host = g.P;
  L->basis_host = g.basis;
  L->pay_host = g.pay_off;
  L->seg_host = g.seg;
  L->side_host = g.side_off;
  *out = L;
  return succeed();
}

kvc_status kvc_append_strided(kvc_layer* L, const void* x, int64_t T, int64_t sb, int64_t sh,
                              int64_t st, void* stream) {
  if (!L) return fail(KVC_ESTATE, "layer is NULL");
  if (T < 0) return fail(KVC_EINVAL, "T must be >= 0");
  if (T == 0) return succeed();
  if (T > L->capacity - L->len)
    return fail(KVC_ECAPACITY, "append of %lld tokens exceeds capacity %lld (length %lld)",
                (long long)T, (long long)L->capacity, (long long)L->len);
  if (!x) return fail(KVC_EINVAL, "x is NULL");
  if (sb < 0 || sh < 0 || st < 0) return fail(KVC_EINVAL, "strides must be >= 0");
  DeviceGuard dg(L->device);
  if (!dg.ok) return fail(KVC_ECUDA, "cannot select the layer's device");
  if (!is_device_ptr(x, L->device)) return fail(KVC_EINVAL, "x is not device memory of the layer's device");
  kvc::AppendArgs a{x, sb, sh, st, T, L->len};
  auto s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  int nk = 0;
  if (L->mode == KVC_MODE_INT8)
    e = kvc::launch_append_int8(L->p, a, s, &nk);
  else if (L->p.prod)
    e = kvc::launch_append_prod(L->p, a, s, &nk);
  else if (L->path == KVC_PATH_AUTO && kvc::tc_append_ok(L->tc, L->p, a))
    e = kvc::launch_append_tc(L->tc, L->p, a, L->wait_ns, s, &nk);
  else if (L->path == KVC_PATH_AUTO && kvc::tc_group_ok(L->tc, L->p, a))
    e = kvc::launch_append_group_tc(L->tc, L->p, a, s, &nk);
  else
    e = kvc::launch_append_generic(L->p, a, s, &nk);
  L->launches += nk;
  if (e != cudaSuccess) return cuda_fail(e, "append launch");
  L->len += T;
  return succeed();
}

kvc_status kvc_append(kvc_layer* L, const void* x, int64_t T, void* stream) {
  if (!L) return fail(KVC_ESTATE, "layer is NULL");
  return kvc_append_strided(L, x, T, (int64_t)L->H * T * L->D, T * (int64_t)L->D, L->D, stream);
}

kvc_status kvc_fetch(kvc_layer* L, void* out, int64_t ld_s, int64_t* S_out, void* stream) {
  if (!L) return fail(KVC_ESTATE, "layer is NULL");
  if (ld_s < L->len) return fail(KVC_EINVAL, "ld_s %lld < length %lld", (long long)ld_s, (long long)L->len);
  if (S_out) *S_out = L->len;
  if (L->len == 0) return succeed();
  if (!out) return fail(KVC_EINVAL, "out is NULL");
  DeviceGuard dg(L->device);
  if (!dg.ok) return fail(KVC_ECUDA, "cannot select the layer's device");
  if (!is_device_ptr(out, L->device)) return fail(KVC_EINVAL, "out is not device memory of the layer's device");
  kvc::FetchArgs f{out, ld_s, L->len};
  auto s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  int nk = 0;
  if (L->mode == KVC_MODE_INT8)
    e = kvc::launch_fetch_int8(L->p, f, s, &nk);
  else if (L->p.prod)
    e = kvc::launch_fetch_prod(L->p, f, s, &nk);
  else if (L->path == KVC_PATH_AUTO && kvc::tc_fetch_ok(L->tc, L->p, f))
    e = kvc::launch_fetch_tc(L->tc, L->p, f, s, &nk);
  else
    e = kvc::launch_fetch_generic(L->p, f, s, &nk);
  L->launches += nk;
  if (e != cudaSuccess) return cuda_fail(e, "fetch launch");
  return succeed();
}

kvc_status kvc_trim(kvc_layer* L, int64_t n, int64_t* dropped) {
  if (!L) return fail(KVC_ESTATE, "layer is NULL");
  int64_t k = std::min(L->len, n);
  if (k < 0) k = 0;
  L->len -= k;
  if (dropped) *dropped = k;
  return succeed();
}

kvc_status kvc_length(const kvc_layer* L, int64_t* out) {
  if (!L) return fail(KVC_ESTATE, "layer is NULL");
  if (!out) return fail(KVC_EINVAL, "out is NULL");
  *out = L->len;
  return succeed();
}

kvc_status kvc_nbytes(const kvc_layer* L, kvc_bytes* out) {
  if (!L) return fail(KVC_ESTATE, "layer is NULL");
  if (!out) return fail(KVC_EINVAL, "out is NULL");
  int64_t payload = 0;
  for (int s = 0; s < L->n_slots; ++s)
    payload += L->len * (L->mode == KVC_MODE_INT8 ? L->D : L->P_host[L->basis_host[s]]);
  out->payload = payload;
  out->side = (int64_t)L->n_slots * L->len * L->side_bytes;
  out->fixed = L->fixed_bytes;
  out->fp16_equiv = (int64_t)L->B * L->H * L->len * L->D * 2;
  return succeed();
}

kvc_status kvc_get_slot_layout(const kvc_layer* L, int32_t slot, kvc_slot_layout* out) {
  if (!L) return fail(KVC_ESTATE, "layer is NULL");
  if (!out) return fail(KVC_EINVAL, "out is NULL");
  if (slot < 0 || slot >= L->n_slots) return fail(KVC_EINVAL, "slot %d outside [0, %d)", slot, L->n_slots);
  out->payload_offset = L->pay_host[slot];
  out->row_bytes = L->mode == KVC_MODE_INT8 ? L->D : L->P_host[L->basis_host[slot]];
  out->side_offset = L->side_host[slot];
  out->side_bytes = L->side_bytes;
  return succeed();
}

kvc_status kvc_set_path(kvc_layer* L, int32_t path) {
  if (!L) return fail(KVC_ESTATE, "layer is NULL");
  if (path != KVC_PATH_AUTO && path != KVC_PATH_GENERIC) return fail(KVC_EINVAL, "unknown path %d", path);
  L->path = path;
  return succeed();
}

}  // extern "C"

namespace {

// Checks shared by the attention entry points; fills the shape fields of a.
kvc_status attend_check(const kvc_layer* K, const kvc_layer* V, int32_t Hq, kvc::AttendArgs& a,
                        size_t* ws_bytes) {
  if (!K || !V) return fail(KVC_ESTATE, "key or value layer is NULL");
  if (K->mode != KVC_MODE_UNIFORM && K->mode != KVC_MODE_CODEBOOK)
    return fail(KVC_EINVAL, "keys must be a uniform or codebook layer");
  if (V->mode != KVC_MODE_INT8 && V->mode != KVC_MODE_UNIFORM)
    return fail(KVC_EINVAL, "values must be an int8 or uniform layer");
  if (K->hpg != 1 || V->hpg != 1) return fail(KVC_EINVAL, "head groups are not supported here");
  if (V->p.prod) return fail(KVC_EINVAL, "values must be an int8 or uniform layer");
  if (K->B != V->B || K->H != V->H || K->D != V->D)
    return fail(KVC_EINVAL, "key and value layers differ in B, H or D");
  if (K->device != V->device) return fail(KVC_EINVAL, "key and value layers are on different devices");
  if (K->len != V->len) return fail(KVC_EINVAL, "key and value layers hold different lengths");
  if (!(K->D == 64 || K->D == 128 || K->D == 256)) return fail(KVC_EINVAL, "D must be 64, 128 or 256");
  if (Hq < K->H || Hq % K->H) return fail(KVC_EINVAL, "Hq must be a multiple of H");
  const int rep = Hq / K->H;
  if (!(rep == 1 || rep == 2 || rep == 4 || rep == 8))
    return fail(KVC_EINVAL, "Hq / H must be 1, 2, 4 or 8");
  if (K->ncpos > 256 || (V->mode == KVC_MODE_UNIFORM && V->ncpos > 256))
    return fail(KVC_EINVAL, "more than 256 packed positions");
  a.Hq = Hq;
  a.rep = rep;
  a.S = K->len;
  a.NCk = std::max(8, K->ncpos);
  a.Dv = V->mode == KVC_MODE_INT8 ? V->D : std::max(8, V->ncpos);
  a.Pk_max = K->pmax;
  a.Pv_max = V->pmax;
  a.out_bf16 = V->p.out_dtype == KVC_BF16 ? 1 : 0;
  int sms = 1;
  {
    DeviceGuard dg(K->device);
    sms = kvc::sm_count();
  }
  if (K->p.prod) {
    a.prod = 1;
    a.m = K->p.m;
    a.n_out = K->p.n_out;
    a.kcode = K->p.code_bytes;
    a.knw = K->side_bytes / 2;
  }
  *ws_bytes = kvc::attend_plan(K->B, Hq, K->n_slots, rep, std::max<int64_t>(K->len, 1), a.NCk,
                               a.Dv, sms, a.m + a.n_out, &a.splits, &a.span);
  return KVC_OK;
}

}  // namespace

extern "C" {

kvc_status kvc_attend_workspace_bytes(const kvc_layer* K, const kvc_layer* V, int32_t Hq,
                                      size_t* out) {
  if (!out) return fail(KVC_EINVAL, "out is NULL");
  kvc::AttendArgs a;
  size_t n = 0;
  kvc_status st = attend_check(K, V, Hq, a, &n);
  if (st) return st;
  *out = n;
  return succeed();
}

kvc_status kvc_attend(const kvc_layer* K, const kvc_layer* V, const float* q, int32_t Hq,
                      float scale, void* out, void* workspace, size_t workspace_bytes,
                      void* stream) {
  kvc::AttendArgs a;
  size_t need = 0;
  kvc_status st = attend_check(K, V, Hq, a, &need);
  if (st) return st;
  if (!(scale >= 0.f) || !std::isfinite(scale)) return fail(KVC_EINVAL, "scale must be finite and >= 0");
  if (!q || !out) return fail(KVC_EINVAL, "q or out is NULL");
  DeviceGuard dg(K->device);
  if (!dg.ok) return fail(KVC_ECUDA, "cannot select the layer's device");
  if (!is_device_ptr(q, K->device) || !is_device_ptr(out, K->device))
    return fail(KVC_EINVAL, "q and out must be device memory of the layers' device");
  auto s = static_cast<cudaStream_t>(stream);
  if (K->len == 0) {  // no stored token: the output is zero
    const cudaError_t e = cudaMemsetAsync(out, 0, (size_t)K->B * Hq * K->D * 2, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(out)");
    return succeed();
  }
  if (!workspace || workspace_bytes < need)
    return fail(KVC_EINVAL, "workspace is NULL or below kvc_attend_workspace_bytes()");
  if (!is_device_ptr(workspace, K->device)) return fail(KVC_EINVAL, "workspace is not device memory");
  if ((uintptr_t)workspace % 256) return fail(KVC_EINVAL, "workspace must be 256-byte aligned");
  a.q = q;
  a.out = out;
  const double sc = scale > 0.f ? (double)scale : 1.0 / std::sqrt((double)K->D);
  a.scale_log2 = (float)(sc * 1.4426950408889634);
  int nk = 0;
  const cudaError_t e = kvc::launch_attend(K->p, V->p, a, workspace, s, &nk);
  const_cast<kvc_layer*>(K)->launches += nk;
  if (e != cudaSuccess) return cuda_fail(e, "attend launch");
  return succeed();
}

kvc_status kvc_code_histogram_bytes(const kvc_layer* L, size_t* out) {
  if (!L) return fail(KVC_ESTATE, "layer is NULL");
  if (!out) return fail(KVC_EINVAL, "out is NULL");
  if (L->mode == KVC_MODE_INT8) return fail(KVC_EINVAL, "int8 layers store no codes");
  if (L->p.prod) return fail(KVC_EINVAL, "the code histogram takes layers without a sketch or outlier stream");
  *out = kvc::histogram_bytes(L->n_slots, std::max(8, L->ncpos));
  return succeed();
}

kvc_status kvc_code_histogram(kvc_layer* L, uint32_t* counts, size_t counts_bytes, void* stream) {
  size_t need = 0;
  kvc_status st = kvc_code_histogram_bytes(L, &need);
  if (st) return st;
  if (!counts || counts_bytes < need) return fail(KVC_EINVAL, "counts is NULL or too small");
  DeviceGuard dg(L->device);
  if (!dg.ok) return fail(KVC_ECUDA, "cannot select the layer's device");
  if (!is_device_ptr(counts, L->device)) return fail(KVC_EINVAL, "counts is not device memory");
  if ((uintptr_t)counts % 4) return fail(KVC_EINVAL, "counts must be 4-byte aligned");
  int nk = 0;
  const cudaError_t e = kvc::launch_code_histogram(L->p, counts, std::max(8, L->ncpos), L->len,
                                                   static_cast<cudaStream_t>(stream), &nk);
  L->launches += nk;
  if (e != cudaSuccess) return cuda_fail(e, "histogram launch");
  return succeed();
}

kvc_status kvc_entropy_bytes(const kvc_layer* L, const uint32_t* counts, kvc_entropy* out) {
  if (!L) return fail(KVC_ESTATE, "layer is NULL");
  if (!counts || !out) return fail(KVC_EINVAL, "counts or out is NULL");
  if (L->mode == KVC_MODE_INT8) return fail(KVC_EINVAL, "int8 layers store no codes");
  if (L->p.prod) return fail(KVC_EINVAL, "the code histogram takes layers without a sketch or outlier stream");
  const int NC = std::max(8, L->ncpos);
  int64_t pre = 0, stored = 0;
  for (int s = 0; s < L->n_slots; ++s) {
    const int b = L->basis_host[s];
    const int64_t fixed = L->len * L->P_host[b];
    int64_t bits = 0, table = 0;
    int nch = 0;
    for (int sg = 0; sg < kvc::kMaxSeg; ++sg) {
      const int32_t* e = &L->seg_host[((size_t)b * kvc::kMaxSeg + sg) * 4];
      if (!e[3]) break;
      const int w = e[1], n = 1 << w;
      for (int m = 0; m < e[3]; ++m) {
        const uint32_t* c = counts + ((size_t)s * NC + nch * 8 + m) * 256;
        const std::vector<int> len = kvc::huffman_code_lengths(c, n);
        for (int v = 0; v < n; ++v) bits += (int64_t)c[v] * len[v];
        table += n;
      }
      nch += (e[3] + 7) / 8;
    }
    const int64_t coded = L->len ? (bits + 7) / 8 + table : 0;
    pre += fixed;
    stored += std::min(fixed, coded);
  }
  out->pre_entropy = pre;
  out->stored_payload = stored;
  out->params = L->fixed_bytes;
  const int64_t total = stored + L->fixed_bytes;
  out->gain = total ? (double)pre / (double)total : 1.0;
  return succeed();
}

// Validate a fit descriptor into FitArgs (choices sorted and distinct, the
// budget clamped to max(choices) * r, beyond which the allocation is the same).
static kvc_status fit_check(const kvc_fit_desc* d, kvc::FitArgs& f) {
  if (!d) return fail(KVC_EINVAL, "descriptor is NULL");
  if (d->in_dtype != KVC_F32 && d->in_dtype != KVC_F16 && d->in_dtype != KVC_BF16)
    return fail(KVC_EINVAL, "in_dtype must be KVC_F32, KVC_F16 or KVC_BF16");
  if (d->B < 1 || d->H < 1) return fail(KVC_EINVAL, "B and H must be >= 1");
  if (d->D < 8 || d->D > kvc::kFitMaxD || d->D % 8)
    return fail(KVC_EINVAL, "D must be a multiple of 8 in [8, %d]", kvc::kFitMaxD);
  if (d->S_fit < 2) return fail(KVC_EINVAL, "the fit needs S_fit >= 2 rows");
  if (d->r < 1 || d->r > d->D) return fail(KVC_EINVAL, "r must be in [1, D]");
  if (!d->bit_choices || d->n_choices < 1 || d->n_choices > kvc::kFitMaxChoices)
    return fail(KVC_EINVAL, "bit_choices must hold 1 .. %d widths", kvc::kFitMaxChoices);
  std::vector<int> ch(d->bit_choices, d->bit_choices + d->n_choices);
  for (int b : ch)
    if (b < 0 || b > 8 || b == 5 || b == 6 || b == 7)
      return fail(KVC_EINVAL, "bit widths must be in {0,1,2,3,4,8}");
  std::sort(ch.begin(), ch.end());
  ch.erase(std::unique(ch.begin(), ch.end()), ch.end());
  if (d->bit_budget < 0 || (int64_t)ch.front() * d->r > d->bit_budget)
    return fail(KVC_EINVAL, "no allocation fits bit_budget with these widths");
  f.x = d->x;
  f.dtype = d->in_dtype;
  f.B = d->B;
  f.H = d->H;
  f.D = d->D;
  f.r = d->r;
  f.S = d->S_fit;
  f.sb = d->stride_b;
  f.sh = d->stride_h;
  f.st = d->stride_t;
  f.n_choices = (int)ch.size();
  for (size_t i = 0; i < ch.size(); ++i) f.choices[i] = ch[i];
  f.budget = (int)std::min<int64_t>(d->bit_budget, (int64_t)ch.back() * d->r);
  f.V = d->V;
  f.mean = d->mean;
  f.bits = d->bits;
  f.qmin = d->qmin;
  f.qstep = d->qstep;
  f.lam_out = d->lam;
  return KVC_OK;
}

kvc_status kvc_fit_uniform_workspace_bytes(const kvc_fit_desc* d, size_t* out) {
  kvc::FitArgs f;
  const kvc_status st = fit_check(d, f);
  if (st) return st;
  if (!out) return fail(KVC_EINVAL, "out is NULL");
  *out = kvc::fit_workspace_bytes(f.B * f.H, f.D, f.r, f.budget);
  return succeed();
}

kvc_status kvc_fit_uniform(const kvc_fit_desc* d, void* workspace, size_t workspace_bytes,
                           void* stream) {
  kvc::FitArgs f;
  const kvc_status st = fit_check(d, f);
  if (st) return st;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  const void* dev_ptrs[] = {f.x, f.V, f.mean, f.bits, f.qmin, f.qstep, workspace};
  for (const void* p : dev_ptrs)
    if (!p || !is_device_ptr(p, dev))
      return fail(KVC_EINVAL, "x, the outputs and the workspace must be device memory of the current device");
  if (f.lam_out && !is_device_ptr(f.lam_out, dev)) return fail(KVC_EINVAL, "lam is not device memory");
  if ((uintptr_t)f.V % 4 || (uintptr_t)f.mean % 4 || (uintptr_t)f.qmin % 4 ||
      (uintptr_t)f.qstep % 4 || (uintptr_t)f.lam_out % 8 ||
      (uintptr_t)f.x % (f.dtype == KVC_F32 ? 4 : 2))
    return fail(KVC_EINVAL, "an array is not aligned to its element size");
  if ((uintptr_t)workspace % 256) return fail(KVC_EINVAL, "workspace must be 256-byte aligned");
  if (workspace_bytes < kvc::fit_workspace_bytes(f.B * f.H, f.D, f.r, f.budget))
    return fail(KVC_EINVAL, "workspace is below kvc_fit_uniform_workspace_bytes()");
  int nk = 0;
  e = kvc::launch_fit_uniform(f, workspace, static_cast<cudaStream_t>(stream), &nk);
  if (e != cudaSuccess) return cuda_fail(e, "fit launch");
  return succeed();
}

kvc_status kvc_fit_outliers(const void* x, int32_t in_dtype, int32_t B, int32_t H, int32_t D,
                            int64_t n_calib, int64_t sb, int64_t sh, int64_t st, int32_t n_out,
                            int32_t* channels, void* stream) {
  if (in_dtype != KVC_F32 && in_dtype != KVC_F16 && in_dtype != KVC_BF16)
    return fail(KVC_EINVAL, "in_dtype must be KVC_F32, KVC_F16 or KVC_BF16");
  if (B < 1 || H < 1 || D < 2 || D > 256) return fail(KVC_EINVAL, "need B, H >= 1 and 2 <= D <= 256");
  if (n_calib < 1) return fail(KVC_EINVAL, "n_calib must be >= 1");
  if (n_out < 1 || n_out > kvc::kProdMaxOut || n_out >= D)
    return fail(KVC_EINVAL, "n_outliers must be in [1, min(%d, D - 1)]", kvc::kProdMaxOut);
  if (sb < 0 || sh < 0 || st < 0) return fail(KVC_EINVAL, "strides must be >= 0");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (!x || !channels || !is_device_ptr(x, dev) || !is_device_ptr(channels, dev))
    return fail(KVC_EINVAL, "x and channels must be device memory of the current device");
  e = kvc::launch_fit_outliers(x, in_dtype, B, H, D, n_calib, sb, sh, st, n_out, channels,
                               static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "outlier fit launch");
  return succeed();
}

kvc_status kvc_set_wait_limit(kvc_layer* L, int64_t ns) {
  if (!L) return fail(KVC_ESTATE, "layer is NULL");
  if (ns < 0) return fail(KVC_EINVAL, "wait limit must be >= 0");
  L->wait_ns = ns == 0 ? kDefaultWaitNs : (uint64_t)ns;
  return succeed();
}

kvc_status kvc_sync_status(kvc_layer* L, void* stream) {
  if (!L) return fail(KVC_ESTATE, "layer is NULL");
  DeviceGuard dg(L->device);
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  int err = 0;
  e = cudaMemcpy(&err, L->p.err, sizeof err, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read error word");
  if (err) {
    e = cudaMemset(L->p.err, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "clear error word");
  }
  if (err == kvc::kErrTimeout) return fail(KVC_ETIMEOUT, "a bounded device wait gave up");
  if (err == kvc::kErrRange) return fail(KVC_EDEVICE, "input outside the exactly encodable range");
  if (err) return fail(KVC_EDEVICE, "device error %d", err);
  return succeed();
}

kvc_status kvc_counters(kvc_layer* L, int64_t out[6], int32_t reset, void* stream) {
  if (!L) return fail(KVC_ESTATE, "layer is NULL");
  if (!out) return fail(KVC_EINVAL, "out is NULL");
  DeviceGuard dg(L->device);
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned long long c[4];
  e = cudaMemcpy(c, L->p.counters, sizeof c, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read counters");
  for (int i = 0; i < 3; ++i) out[i] = (int64_t)c[i];
  out[3] = L->launches;
  float ratio;
  const uint32_t bits = (uint32_t)c[3];
  std::memcpy(&ratio, &bits, sizeof ratio);
  out[4] = (int64_t)std::llround((double)ratio * 1e6);
  out[5] = 0;
  if (reset) {
    L->launches = 0;
    e = cudaMemset(L->p.counters, 0, sizeof c);
    if (e != cudaSuccess) return cuda_fail(e, "clear counters");
  }
  return succeed();
}

void kvc_destroy(kvc_layer* L) {
  if (!L) return;
  {
    DeviceGuard dg(L->device);
    if (L->block) cudaFree(L->block);
    kvc::tc_release(L->tc);
  }
  delete L;
}

}  // extern "C"
