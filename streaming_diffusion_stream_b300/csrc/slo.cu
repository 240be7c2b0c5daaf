// slo.cu -- the SLO-aware stream-batch controller (host code only).
//
// StreamDiffusionV2 summary, "SLO-aware batching scheduler": given a target
// frame rate, the scheduler sizes the stream batch B so that every stream
// meets its deadline while the aggregate rate approaches the roofline knee.
// The latency of an iteration over B*T frames is modelled as affine in
// B*T (activation traffic linear in B*T plus a fixed part), fitted to the
// observed latencies by weighted least squares.
#include <cmath>
#include <vector>

#include "sds_internal.h"

struct sds_slo {
  sds_slo_config cfg;
  struct Obs {
    double x, y, w;  // frames B*T, latency, weight
    int64_t batch;
  };
  std::vector<Obs> obs;
};

namespace {

// Weighted least-squares line y = a + b x; false when x does not vary.
bool fit_line(const std::vector<sds_slo::Obs>& obs, double& a, double& b) {
  double sw = 0, sx = 0, sy = 0;
  for (const auto& o : obs) {
    sw += o.w;
    sx += o.w * o.x;
    sy += o.w * o.y;
  }
  if (sw <= 0) return false;
  const double mx = sx / sw, my = sy / sw;
  double sxx = 0, sxy = 0;
  for (const auto& o : obs) {
    sxx += o.w * (o.x - mx) * (o.x - mx);
    sxy += o.w * (o.x - mx) * (o.y - my);
  }
  if (!(sxx > 0)) return false;
  b = sxy / sxx;
  a = my - b * mx;
  return true;
}

}  // namespace

extern "C" {

sds_status sds_slo_create(const sds_slo_config* cfg, sds_slo** out) {
  if (!out) return SDS_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || !(cfg->target_fps > 0) || !(cfg->forget > 0 && cfg->forget <= 1) ||
      !(cfg->knee_gain >= 0 && cfg->knee_gain < 1) || cfg->frames_T < 1 || cfg->b_min < 1 ||
      cfg->b_max < cfg->b_min) {
    sds::set_thread_error("slo_create: invalid config (target_fps > 0, forget in (0,1], "
                          "knee_gain in [0,1), frames_T >= 1, 1 <= b_min <= b_max)");
    return SDS_ERR_INVALID_ARG;
  }
  sds_slo* c = new sds_slo();
  c->cfg = *cfg;
  *out = c;
  return SDS_OK;
}

void sds_slo_destroy(sds_slo* c) { delete c; }

sds_status sds_slo_observe(sds_slo* c, int64_t batch, double latency_s) {
  if (!c) return SDS_ERR_INVALID_ARG;
  if (batch < 1 || !(latency_s > 0) || !std::isfinite(latency_s)) {
    sds::set_thread_error("slo_observe: need batch >= 1 and a finite latency > 0");
    return SDS_ERR_INVALID_ARG;
  }
  for (auto& o : c->obs) o.w *= c->cfg.forget;
  c->obs.push_back({(double)(batch * c->cfg.frames_T), latency_s, 1.0, batch});
  return SDS_OK;
}

sds_status sds_slo_choose(const sds_slo* c, sds_slo_choice* out) {
  if (!c || !out) return SDS_ERR_INVALID_ARG;
  const sds_slo_config& g = c->cfg;
  sds_slo_choice r{};
  double a = 0, b = 0;
  if (!fit_line(c->obs, a, b)) {
    // explore: the smallest B not observed yet
    int64_t next = g.b_min;
    for (; next < g.b_max; ++next) {
      bool seen = false;
      for (const auto& o : c->obs) seen = seen || o.batch == next;
      if (!seen) break;
    }
    r.batch = next;
    r.exploring = 1;
    *out = r;
    return SDS_OK;
  }
  const double T = (double)g.frames_T;
  auto latency = [&](int64_t B) { return a + b * (double)B * T; };
  auto total = [&](int64_t B) { return (double)B * T / latency(B); };
  int64_t b_slo = 0;
  for (int64_t B = g.b_min; B <= g.b_max; ++B) {
    const double L = latency(B);
    if (L > 0 && T / L >= g.target_fps) b_slo = B;
  }
  const double f_max = total(g.b_max);
  int64_t b_knee = g.b_max;
  for (int64_t B = g.b_min; B <= g.b_max; ++B) {
    if (latency(B) > 0 && total(B) >= (1.0 - g.knee_gain) * f_max) {
      b_knee = B;
      break;
    }
  }
  r.b_slo = b_slo;
  r.b_knee = b_knee;
  r.batch = b_slo > 0 ? (b_slo < b_knee ? b_slo : b_knee) : g.b_min;
  r.a = a;
  r.b = b;
  r.latency_s = latency(r.batch);
  r.per_stream_fps = T / r.latency_s;
  r.total_fps = total(r.batch);
  r.meets_slo = r.per_stream_fps >= g.target_fps ? 1 : 0;
  *out = r;
  return SDS_OK;
}

}  // extern "C"
