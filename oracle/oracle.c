/*
 * oracle.c -- plain, slow CPU oracle for the fused-chain hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the bench's CPU
 * baseline do.  It shares no code, header, table or constant with the CUDA
 * path: it has its own dtype conversions, its own rounding, and its own
 * reading of every formula.
 *
 * Every computation is a scalar loop in IEEE binary64, one operation at a
 * time, in the order the method's pages state it.  Values are converted
 * exactly from their stored dtype (fp16 / bf16 / fp32 -> double) and rounded
 * only where the method rounds (an explicit cast in a chain; the dtype a
 * result is stored in, which the caller applies).
 *
 * Sources followed (page title, section):
 *  - "DeepJIT ... 串行小核墙" (hotelren.com), section 3.2: the add -> relu ->
 *    scale kernel, relu written as t > 0 ? t : 0; section 4.1: a chain of
 *    several inputs (a + b) -> relu -> scale -> + c; section 4.2: the same
 *    chain element by element; section 3.3: sizes baked into the kernel.
 *  - "算子与运行时" (gtnt.cn), section 2: ChannelShuffle as
 *    reshape(n, g, c/g, h, w) -> transpose(1, 2) -> reshape(n, c, h, w);
 *    section 2.3: fp32 accumulation for low-precision data.
 *  - "TeleTron ..." (2kiu.com), section 3.3: residual add + RMSNorm with a
 *    per-row reduction and higher-precision accumulation; section 4.2: the
 *    RMSNorm scale rsqrt(sum_sq / K + 1e-6) (eps inside the root); section
 *    3.1: QKV projection -> head split -> RoPE as one multi-step fusion.
 *  - The detection-head decode (sigmoid, exp/mul/add, slice, concat, cast)
 *    is named in "DeepJIT", section 1.1; its formula is the workload
 *    definition of the detection-head decode benchmark (YOLO-style decode).
 *
 * Where the pages leave a step open, the reading taken is stated at the
 * function that takes it.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { DT_F32 = 0, DT_F16 = 1, DT_BF16 = 2 };

enum {
  OP_ADD = 1,     /* x + in_j           (new input tensor of the current dtype) */
  OP_MUL = 2,     /* x * in_j           (new input tensor of the current dtype) */
  OP_SCALE = 3,   /* x * c              (c an fp32 constant) */
  OP_RELU = 4,    /* x > 0 ? x : 0 */
  OP_SIGMOID = 5, /* 1 / (1 + exp(-x)) */
  OP_EXP = 6,     /* exp(x) */
  OP_CAST = 7,    /* round to dtype (arg), continue in the working type */
  OP_EXP_FAST = 8,    /* exp(x), approximated on the device ("exp:fast") */
  OP_SIGMOID_FAST = 9 /* 1 / (1 + exp(-x)), approximated likewise ("sigmoid:fast") */
};

/* ------------------------------------------------------------------ */
/* dtype conversions, written from the IEEE 754 binary formats           */
/* ------------------------------------------------------------------ */

/* fp16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double f16_bits_to_double(uint16_t h) {
  int s = h >> 15, e = (h >> 10) & 0x1f, m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(m | 0x400), e - 25); /* (1024 + m) * 2^(e - 15 - 10) */
  return s ? -v : v;
}

/* bf16: the upper 16 bits of an fp32. */
static double bf16_bits_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static double load_elem(const void* p, int dt, int64_t i) {
  if (dt == DT_F32) return (double)((const float*)p)[i];
  if (dt == DT_F16) return f16_bits_to_double(((const uint16_t*)p)[i]);
  return bf16_bits_to_double(((const uint16_t*)p)[i]);
}

/* Round x to nearest, ties to even, in a binary format with p significand
 * bits (hidden bit included), smallest normal exponent emin and largest
 * exponent emax.  Results beyond the largest finite value become +-inf,
 * exactly as IEEE round-to-nearest does; subnormals are kept. */
static double round_binary(double x, int p, int emin, int emax) {
  if (isnan(x) || isinf(x) || x == 0.0) return x;
  double ax = fabs(x);
  int e;
  frexp(ax, &e); /* ax = f * 2^e with f in [0.5, 1): leading bit 2^(e-1) */
  int lead = e - 1;
  if (lead < emin) lead = emin; /* subnormal range: fixed quantum */
  double q = ldexp(1.0, lead - (p - 1)); /* one unit in the last place */
  double r = ax / q;                     /* exact: q is a power of two */
  double fl = floor(r);
  double frac = r - fl;
  double n = fl;
  if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) != 0.0)) n = fl + 1.0;
  double res = n * q;
  double maxf = ldexp(2.0 - ldexp(1.0, 1 - p), emax);
  if (res > maxf) res = INFINITY;
  return copysign(res, x);
}

double oracle_round_f16(double x) { return round_binary(x, 11, -14, 15); }
double oracle_round_bf16(double x) { return round_binary(x, 8, -126, 127); }
double oracle_round_f32(double x) { return round_binary(x, 24, -126, 127); }

static double round_to(int dt, double x) {
  if (dt == DT_F16) return oracle_round_f16(x);
  if (dt == DT_BF16) return oracle_round_bf16(x);
  return oracle_round_f32(x);
}

/* Bit pattern of an fp16-representable double (already rounded). */
static uint16_t f16_bits_of(double v) {
  uint16_t s = signbit(v) ? 0x8000 : 0;
  if (isnan(v)) return 0x7e00;
  double a = fabs(v);
  if (isinf(a)) return s | 0x7c00;
  if (a == 0.0) return s;
  if (a < ldexp(1.0, -14)) return s | (uint16_t)(a / ldexp(1.0, -24)); /* subnormal */
  int e;
  double f = frexp(a, &e); /* a = f * 2^e, f in [0.5,1) */
  int biased = e - 1 + 15;
  uint16_t m = (uint16_t)((f * 2.0 - 1.0) * 1024.0);
  return s | (uint16_t)(biased << 10) | m;
}

static uint16_t bf16_bits_of(double v) {
  if (isnan(v)) return 0x7fc0;
  float f = (float)v; /* exact: v is bf16-representable */
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* Store rounded values in a dtype's bit layout (out: float[] or uint16[]). */
void oracle_store(const double* v, int64_t n, int dt, void* out) {
  for (int64_t i = 0; i < n; ++i) {
    double r = round_to(dt, v[i]);
    if (dt == DT_F32)
      ((float*)out)[i] = (float)r;
    else if (dt == DT_F16)
      ((uint16_t*)out)[i] = f16_bits_of(r);
    else
      ((uint16_t*)out)[i] = bf16_bits_of(r);
  }
}

/* Exact conversion of stored values to double (for tests of the pins). */
void oracle_load(const void* p, int dt, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = load_elem(p, dt, i);
}

/* ------------------------------------------------------------------ */
/* Elementwise chains                                                   */
/* ------------------------------------------------------------------ */

/* The working type of a fused chain is fp32 (the pages keep elementwise
 * steps in high precision in registers and round only at casts and at the
 * final store).  The oracle computes in binary64 but keeps the fp32 RANGE:
 * a magnitude at or above the fp32 overflow threshold (the largest finite
 * fp32 plus half an ulp, 2^128 - 2^103) is infinity, as it is on the device.
 */
static const double FP32_OVF = 340282356779733661637539395458142568448.0; /* 2^128 - 2^103 */

static double fp32_range(double v) {
  if (!isnan(v) && fabs(v) >= FP32_OVF) return copysign(INFINITY, v);
  return v;
}

/* One op of a chain on an exact value x; b is the op's input tensor element
 * (add/mul), c the op's constant (scale) or target dtype (cast). */
static double apply_op(int op, double x, double b, double c) {
  switch (op) {
    case OP_ADD: return x + b;
    case OP_MUL: return x * b;
    case OP_SCALE: return x * c;
    case OP_RELU: return x > 0.0 ? x : 0.0; /* NaN and -0 give +0 */
    case OP_SIGMOID:
    case OP_SIGMOID_FAST: return 1.0 / (1.0 + exp(-x));
    case OP_EXP:
    case OP_EXP_FAST: return exp(x);
    case OP_CAST: return round_to((int)c, x);
    default: return NAN;
  }
}

/* Index of input 0 for output element e when the chain starts with a
 * ChannelShuffle of `groups` groups on an NCHW tensor: the output channel
 * co = j*groups + i holds input channel ci = i*(C/groups) + j
 * (reshape (n, g, C/g, h, w), swap axes 1 and 2, reshape back). */
static int64_t shuffle_src(int64_t e, int groups, const int64_t* nchw) {
  int64_t C = nchw[1], HW = nchw[2] * nchw[3];
  int64_t n = e / (C * HW), co = (e / HW) % C, hw = e % HW;
  int64_t cpg = C / groups;
  int64_t j = co / groups, i = co % groups;
  int64_t ci = i * cpg + j;
  return (n * C + ci) * HW + hw;
}

/*
 * Plain evaluation of a chain.
 *   ops[k], args[k]    : op code and constant (scale value as an fp32, or the
 *                        cast's target dtype)
 *   in_idx[k]          : for add/mul, which input tensor the op consumes
 *   inputs[j], in_dt[j]: input tensors and their stored dtypes
 *   idx (may be NULL)  : output element indices to evaluate (else 0..n-1)
 *   groups/nchw        : groups > 0 prefixes the chain with a ChannelShuffle
 *                        of input 0 on the NCHW shape nchw
 *   out                : exact (binary64) result of each element before the
 *                        final store; the caller rounds it to the output dtype
 */
void oracle_chain_eval(int n_ops, const int* ops, const double* args, const int* in_idx,
                       const void* const* inputs, const int* in_dt, int64_t n_out,
                       const int64_t* idx, int groups, const int64_t* nchw, double* out) {
  for (int64_t s = 0; s < n_out; ++s) {
    int64_t e = idx ? idx[s] : s;
    int64_t e0 = groups > 0 ? shuffle_src(e, groups, nchw) : e;
    double x = load_elem(inputs[0], in_dt[0], e0);
    for (int k = 0; k < n_ops; ++k) {
      double b = 0.0;
      if (ops[k] == OP_ADD || ops[k] == OP_MUL) b = load_elem(inputs[in_idx[k]], in_dt[in_idx[k]], e);
      x = fp32_range(apply_op(ops[k], x, b, args[k]));
    }
    out[s] = x;
  }
}

/*
 * Acceptance check for a device result of a chain (test helper).
 *
 * Two rules, tried in order:
 *  (1) the flat tolerance of the output dtype against the plain value:
 *      fp32 1e-6 relative, fp16 at most 2 ulp from the correctly rounded
 *      value, bf16 8e-3 relative; inf must match in sign, NaN matches NaN;
 *  (2) a first-order running error bound (running error analysis in the
 *      sense of Wilkinson): alongside the exact value v of each step the
 *      check carries a bound E on |device - v| for a device that evaluates
 *      every step in IEEE fp32:
 *        add/mul/scale:  E' = |m|E(1+u) + u|v'| + eta   (m = 1, b or c)
 *        relu:           E' = E                          (1-Lipschitz, exact)
 *        exp:            E' = e^v (e^E - 1) + 4u e^(v+E) + eta
 *                        (expf is documented to 2 ulp = 4u relative)
 *        sigmoid:        E' = D E + 10u (sigma(v) + D E) + eta
 *                        (D the largest |sigma'| on [v - E, v + E], at most
 *                        1/4; expf 2 ulp, the add 1/2 ulp, the reciprocal
 *                        within 1 ulp, with margin), widened to
 *                        [0, sigma(v + E)] where 1 + exp(-x) can reach 2^126
 *        exp:fast:       E' = e^v (e^E - 1) + (1.25 (|v| + E) + 3) u e^(v+E)
 *                        + 2^-126 + eta
 *                        (the device forms x * L with L the fp32 nearest log2 e:
 *                        the product's rounding and L's are 1.25 u |x| in the
 *                        exponent, a relative 1.25 u |x| in the result; the
 *                        hardware 2^t is within 3 u relative; results below
 *                        2^-126 flush to zero)
 *        sigmoid:fast:   as sigmoid, with (1.25 (|v| + E) + 9) u in place of
 *                        10 u (the fast exp's relative error reaches the
 *                        sigmoid at most in full, plus the add and the
 *                        reciprocal, with margin)
 *      with u = 2^-24 and eta = 2^-147 covering fp32 underflow.  Where the
 *      interval [v - E, v + E] straddles a rounding boundary of a cast or the
 *      fp32 overflow threshold, each outcome is followed as its own branch;
 *      more than MAXB live branches make the element "unpinned".
 *
 * gpu_out holds the device output in out_dt's bit layout.  class_out[s]
 * (may be NULL) gets 0 = flat pass, 1 = pass by the error bound, 2 = fail,
 * 3 = unpinned.  Returns the number of failures; counts[0..3] gets the
 * number of elements in each class.
 */
#define MAXB 16
typedef struct {
  double v, e;
} branch_t;

static const double U32 = 5.9604644775390625e-08; /* 2^-24 */
static const double ETA = 5.605193857299268e-45;  /* 2^-147 */
static const double FTZ32 = 1.1754943508222875e-38; /* 2^-126: flush-to-zero */

static int f16_order(uint16_t h) { /* monotone integer image of an fp16 */
  return (h & 0x8000) ? -(int)(h & 0x7fff) : (int)h;
}

static int is_inf_or_nan(double v) { return isnan(v) || isinf(v); }

/* Apply one op to a branch; writes 1 or 2 successor branches. */
static int step_branch(int op, branch_t s, double b, double c, int out_dt_unused, branch_t* nb) {
  (void)out_dt_unused;
  double v = s.v, E = s.e, vn, En;
  if (is_inf_or_nan(v)) { /* exact IEEE semantics from here on */
    nb[0].v = fp32_range(apply_op(op, v, b, c));
    nb[0].e = 0.0;
    return 1;
  }
  switch (op) {
    case OP_ADD:
      vn = v + b;
      En = E * (1 + U32) + U32 * fabs(vn) + ETA;
      break;
    case OP_MUL:
      vn = v * b;
      En = fabs(b) * E * (1 + U32) + U32 * fabs(vn) + ETA;
      break;
    case OP_SCALE:
      vn = v * c;
      En = fabs(c) * E * (1 + U32) + U32 * fabs(vn) + ETA;
      break;
    case OP_RELU:
      vn = v > 0.0 ? v : 0.0;
      En = E;
      break;
    case OP_EXP:
      vn = exp(v);
      En = vn * expm1(E) + 4 * U32 * exp(v + E) + ETA;
      break;
    case OP_EXP_FAST:
      vn = exp(v);
      En = vn * expm1(E) + (1.25 * (fabs(v) + E) + 3) * U32 * exp(v + E) + FTZ32 + ETA;
      break;
    case OP_SIGMOID:
    case OP_SIGMOID_FAST: {
      /* the relative error of the device's exp, add and reciprocal */
      const double c = op == OP_SIGMOID ? 10.0 : 1.25 * (fabs(v) + E) + 9.0;
      vn = 1.0 / (1.0 + exp(-v));
      /* |sigma'(x)| = sigma(x)(1 - sigma(x)) is largest at x = 0: take its
         maximum over [v - E, v + E] (mean value theorem) */
      double xm = (v - E <= 0.0 && v + E >= 0.0) ? 0.0 : (v > 0.0 ? v - E : v + E);
      double sm = 1.0 / (1.0 + exp(-xm));
      double dmax = sm * (1.0 - sm);
      En = dmax * E + c * U32 * (vn + dmax * E) + ETA;
      /* from -x >= 87 on, 1 + exp(-x) may reach 2^126 (or overflow to inf) in
         fp32 and the device's reciprocal returns 0 for a true value below
         2^-126: accept any value in [0, sigma(v + E)] there */
      if (-(v - E) >= 87.0) {
        double hi = 1.0 / (1.0 + exp(-(v + E)));
        if (hi * (1 + c * U32) > En) En = hi * (1 + c * U32) + ETA;
      }
      break;
    }
    case OP_CAST: {
      int dt = (int)c;
      if (dt == DT_F32) {
        /* the device value is already fp32 and stays as it is, while the
           exact value is rounded: |g - round32(v)| <= E + u|v| */
        vn = round_to(DT_F32, v);
        En = E + U32 * fabs(v);
        break;
      }
      double lo = round_to(dt, v - E), hi = round_to(dt, v + E);
      if (E == 0.0 || lo == hi) {
        nb[0].v = fp32_range(round_to(dt, v));
        nb[0].e = 0.0;
        return 1;
      }
      /* the device value rounds to one of the representable values in
         [lo, hi] (rounding is monotone): follow each of them */
      int olo = f16_order(dt == DT_F16 ? f16_bits_of(lo) : bf16_bits_of(lo));
      int ohi = f16_order(dt == DT_F16 ? f16_bits_of(hi) : bf16_bits_of(hi));
      if (ohi - olo + 1 > MAXB) return -1;
      int nn = 0;
      for (int o = olo; o <= ohi; ++o) {
        uint16_t bits = o >= 0 ? (uint16_t)o : (uint16_t)(0x8000 | (-o));
        nb[nn].v = fp32_range(dt == DT_F16 ? f16_bits_to_double(bits) : bf16_bits_to_double(bits));
        nb[nn].e = 0.0;
        ++nn;
      }
      return nn;
    }
    default:
      return -1;
  }
  /* the fp32 overflow threshold */
  if (!isnan(vn) && fabs(vn) + En >= FP32_OVF && fabs(vn) - En < FP32_OVF) {
    nb[0].v = vn;
    nb[0].e = En;
    nb[1].v = copysign(INFINITY, vn);
    nb[1].e = 0.0;
    return 2;
  }
  nb[0].v = fp32_range(vn);
  nb[0].e = is_inf_or_nan(nb[0].v) ? 0.0 : En;
  return 1;
}

static double device_value(const void* p, int dt, int64_t s) { return load_elem(p, dt, s); }

static int flat_pass(double g, uint16_t gbits, double r, int out_dt) {
  if (isnan(r) || isnan(g)) return isnan(r) && isnan(g);
  if (isinf(r)) return g == r;
  if (out_dt == DT_F16) { /* distance in ulps from the correctly rounded value */
    int d = f16_order(gbits) - f16_order(f16_bits_of(oracle_round_f16(r)));
    if (d < 0) d = -d;
    return d <= 2;
  }
  if (isinf(g)) return 0;
  if (out_dt == DT_F32) return fabs(g - r) <= 1e-6 * fabs(r);
  return fabs(g - r) <= 8e-3 * fabs(r); /* bf16 */
}

static int bound_pass(double g, branch_t s, int out_dt) {
  if (isnan(s.v)) return isnan(g);
  if (isinf(s.v)) return g == s.v;
  if (isnan(g)) return 0;
  if (out_dt == DT_F32) return fabs(g - s.v) <= s.e;
  /* the final store rounds: any rounding of a value in [v-E, v+E] */
  double lo = round_to(out_dt, s.v - s.e), hi = round_to(out_dt, s.v + s.e);
  return g >= lo && g <= hi;
}

int64_t oracle_chain_check(int n_ops, const int* ops, const double* args, const int* in_idx,
                           const void* const* inputs, const int* in_dt, int64_t n_out,
                           const int64_t* idx, int groups, const int64_t* nchw,
                           const void* gpu_out, int out_dt, int8_t* class_out, int64_t* counts) {
  int64_t fails = 0;
  for (int c = 0; c < 4; ++c) counts[c] = 0;
  for (int64_t s = 0; s < n_out; ++s) {
    int64_t e = idx ? idx[s] : s;
    int64_t e0 = groups > 0 ? shuffle_src(e, groups, nchw) : e;
    double g = device_value(gpu_out, out_dt, s);
    uint16_t gbits = out_dt == DT_F32 ? 0 : ((const uint16_t*)gpu_out)[s];

    /* rule 1: flat tolerance against the plain value */
    double x = load_elem(inputs[0], in_dt[0], e0);
    for (int k = 0; k < n_ops; ++k) {
      double b = 0.0;
      if (ops[k] == OP_ADD || ops[k] == OP_MUL) b = load_elem(inputs[in_idx[k]], in_dt[in_idx[k]], e);
      x = fp32_range(apply_op(ops[k], x, b, args[k]));
    }
    int cls;
    if (flat_pass(g, gbits, x, out_dt)) {
      cls = 0;
    } else {
      /* rule 2: running error bound with branches */
      branch_t cur[MAXB], nxt[MAXB * MAXB];
      int nc = 1, unpinned = 0;
      cur[0].v = load_elem(inputs[0], in_dt[0], e0);
      cur[0].e = 0.0;
      for (int k = 0; k < n_ops && !unpinned; ++k) {
        double b = 0.0;
        if (ops[k] == OP_ADD || ops[k] == OP_MUL) b = load_elem(inputs[in_idx[k]], in_dt[in_idx[k]], e);
        int nn = 0;
        for (int i = 0; i < nc; ++i) {
          int r = step_branch(ops[k], cur[i], b, args[k], out_dt, nxt + nn);
          if (r < 0) { unpinned = 1; break; }
          nn += r;
        }
        if (nn > MAXB) unpinned = 1;
        if (!unpinned) {
          memcpy(cur, nxt, sizeof(branch_t) * (size_t)nn);
          nc = nn;
        }
      }
      if (unpinned) {
        cls = 3;
      } else {
        cls = 2;
        for (int i = 0; i < nc; ++i)
          if (bound_pass(g, cur[i], out_dt)) { cls = 1; break; }
      }
    }
    if (cls == 2) ++fails;
    counts[cls]++;
    if (class_out) class_out[s] = (int8_t)cls;
  }
  return fails;
}

/* ------------------------------------------------------------------ */
/* ChannelShuffle                                                       */
/* ------------------------------------------------------------------ */

/* out[n, j*g + i, :, :] = in[n, i*(C/g) + j, :, :] for i < g, j < C/g,
 * copied byte for byte (elem_bytes per element). */
void oracle_channel_shuffle(const void* in, void* out, int64_t n, int64_t c, int64_t h, int64_t w,
                            int groups, int elem_bytes) {
  int64_t hw = h * w, cpg = c / groups;
  const char* src = (const char*)in;
  char* dst = (char*)out;
  for (int64_t b = 0; b < n; ++b)
    for (int64_t i = 0; i < groups; ++i)
      for (int64_t j = 0; j < cpg; ++j) {
        int64_t co = j * groups + i, ci = i * cpg + j;
        for (int64_t p = 0; p < hw; ++p) {
          int64_t so = ((b * c + ci) * hw + p) * elem_bytes;
          int64_t dO = ((b * c + co) * hw + p) * elem_bytes;
          memcpy(dst + dO, src + so, (size_t)elem_bytes);
        }
      }
}

/* ------------------------------------------------------------------ */
/* Residual add + RMSNorm                                               */
/* ------------------------------------------------------------------ */

/* For each row: h = x + residual; residual_out = h; ms = sum(h^2) / hidden;
 * y = h * (1 / sqrt(ms + eps)) * w.  All in binary64; eps is the fp32 value
 * the caller passes (inside the square root, as the pages write it).
 * Reading: the statistics are taken on the unrounded sum h, and the updated
 * residual is h stored in the activation dtype. */
void oracle_rmsnorm_residual(const void* x, const void* res, const void* w, int dt, int64_t rows,
                             int64_t hidden, float eps, double* y, double* res_out) {
  for (int64_t r = 0; r < rows; ++r) {
    double ms = 0.0;
    for (int64_t k = 0; k < hidden; ++k) {
      double hk = load_elem(x, dt, r * hidden + k) + load_elem(res, dt, r * hidden + k);
      res_out[r * hidden + k] = hk;
      ms += hk * hk;
    }
    ms /= (double)hidden;
    double rstd = 1.0 / sqrt(ms + (double)eps);
    for (int64_t k = 0; k < hidden; ++k)
      y[r * hidden + k] = res_out[r * hidden + k] * rstd * load_elem(w, dt, k);
  }
}

/* ------------------------------------------------------------------ */
/* RMSNorm feeding a Linear layer, then an elementwise scale             */
/* ------------------------------------------------------------------ */

/* "TeleTron" section 4.2 (RMSNorm + Linear + scale): per row m of x [M, K]
 *   s_m = 1 / sqrt(sum_k x[m,k]^2 / K + eps)          (the RMSNorm factor)
 *   out[m, n] = scale * (sum_k x[m,k] * s_m * gamma[k] * w[n,k] + bias[n])
 * with w in [N, K] (the transposed layout the page recommends for the
 * weight).  Reading: the statistics are taken on x, as RMSNorm defines them
 * (the page's pseudo-code squares x * gamma).  rows: the row indices to
 * evaluate (nrows of them); out and mag are [nrows, N]; mag gets
 * |scale| * (s_m * sum_k |x gamma w| + |bias|), the scale of the terms. */
void oracle_rmsnorm_linear(const void* x, const void* gamma, const void* w, const void* bias,
                           int dt, int64_t K, int64_t N, const int64_t* rows, int64_t nrows,
                           float eps, float scale, double* out, double* mag) {
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t m = rows[i];
    double ss = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      double v = load_elem(x, dt, m * K + k);
      ss += v * v;
    }
    double s = 1.0 / sqrt(ss / (double)K + (double)eps);
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0, absacc = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        double t = load_elem(x, dt, m * K + k) * s * load_elem(gamma, dt, k) *
                   load_elem(w, dt, n * K + k);
        acc += t;
        absacc += fabs(t);
      }
      double b = bias ? load_elem(bias, dt, n) : 0.0;
      out[i * N + n] = (double)scale * (acc + b);
      if (mag) mag[i * N + n] = fabs((double)scale) * (absacc + fabs(b));
    }
  }
}

/* ------------------------------------------------------------------ */
/* Residual add + LayerNorm                                             */
/* ------------------------------------------------------------------ */

/* "DeepJIT" section 4.3 (one block per row): mean = sum(h)/n,
 * var = sum(h^2)/n - mean^2, y = (h - mean) / sqrt(var + eps) * gamma + beta,
 * here with h = x + residual.  res, gamma, beta may be NULL (no residual,
 * gamma = 1, beta = 0).  res_out receives h when res is given.  mag receives,
 * per output, the sum of the magnitudes of the terms of
 * y = h*s*gamma - mean*s*gamma + beta (s = 1/sqrt(var + eps)), where the
 * mean is itself a sum of the hidden terms h_k / hidden, whose magnitudes
 * add up to mean(|h|):  mag = (|h| + mean(|h|)) * s * |gamma| + |beta|. */
void oracle_layernorm_residual(const void* x, const void* res, const void* gamma, const void* beta,
                               int dt, int64_t rows, int64_t hidden, float eps, double* y,
                               double* res_out, double* mag) {
  for (int64_t r = 0; r < rows; ++r) {
    double s1 = 0.0, s2 = 0.0, sa = 0.0;
    for (int64_t k = 0; k < hidden; ++k) {
      double hk = load_elem(x, dt, r * hidden + k);
      if (res) hk += load_elem(res, dt, r * hidden + k);
      if (res_out) res_out[r * hidden + k] = hk;
      s1 += hk;
      s2 += hk * hk;
      sa += fabs(hk);
    }
    double mean = s1 / (double)hidden, mean_abs = sa / (double)hidden;
    double var = s2 / (double)hidden - mean * mean;
    double s = 1.0 / sqrt(var + (double)eps);
    for (int64_t k = 0; k < hidden; ++k) {
      double hk = load_elem(x, dt, r * hidden + k);
      if (res) hk += load_elem(res, dt, r * hidden + k);
      double g = gamma ? load_elem(gamma, dt, k) : 1.0;
      double b = beta ? load_elem(beta, dt, k) : 0.0;
      y[r * hidden + k] = (hk - mean) * s * g + b;
      if (mag) mag[r * hidden + k] = (fabs(hk) + mean_abs) * s * fabs(g) + fabs(b);
    }
  }
}

/* ------------------------------------------------------------------ */
/* QKV split + transpose + rotate-half RoPE                             */
/* ------------------------------------------------------------------ */

/* qkv is [tokens, 3, heads, D] (q block, k block, v block per token).
 * Outputs are [heads, tokens, D].  Token t sits at position pos[t].
 * For i < D/2: theta = pos * base^(-2i/D);
 *   o[i]       = x[i] cos(theta) - x[i + D/2] sin(theta)
 *   o[i + D/2] = x[i + D/2] cos(theta) + x[i] sin(theta)
 * on q and k; v is copied.  term_mag (may be NULL) receives, per q/k output,
 * |first term| + |second term| (the scale the tolerance is relative to). */
void oracle_rope_qkv_split(const void* qkv, int dt, int64_t tokens, int heads, int D,
                           const int64_t* pos, double base, double* q, double* k, double* v,
                           double* q_mag, double* k_mag) {
  int half = D / 2;
  for (int64_t t = 0; t < tokens; ++t) {
    for (int which = 0; which < 3; ++which) {
      double* dst = which == 0 ? q : which == 1 ? k : v;
      double* mag = which == 0 ? q_mag : which == 1 ? k_mag : NULL;
      for (int h = 0; h < heads; ++h) {
        int64_t src = ((t * 3 + which) * heads + h) * (int64_t)D;
        int64_t out = ((int64_t)h * tokens + t) * D;
        if (which == 2) {
          for (int d = 0; d < D; ++d) dst[out + d] = load_elem(qkv, dt, src + d);
          continue;
        }
        for (int i = 0; i < half; ++i) {
          double theta = (double)pos[t] * pow(base, -2.0 * i / D);
          double c = cos(theta), s = sin(theta);
          double x1 = load_elem(qkv, dt, src + i), x2 = load_elem(qkv, dt, src + i + half);
          dst[out + i] = x1 * c - x2 * s;
          dst[out + i + half] = x2 * c + x1 * s;
          if (mag) {
            mag[out + i] = fabs(x1 * c) + fabs(x2 * s);
            mag[out + i + half] = fabs(x2 * c) + fabs(x1 * s);
          }
        }
      }
    }
  }
}

/* ------------------------------------------------------------------ */
/* Detection-head decode                                                */
/* ------------------------------------------------------------------ */

/* feats[s] is [1, na*no, H_s, W_s]; channel a*no + k.  For each scale s,
 * anchor a, cell (y, x), channel k: p = sigmoid(feat);
 *   k = 0: (2p - 0.5 + x) * stride_s      k = 1: (2p - 0.5 + y) * stride_s
 *   k = 2: (2p)^2 * anchor_w[s][a]        k = 3: (2p)^2 * anchor_h[s][a]
 *   k >= 4: p
 * written to out[row, k] with row = off_s + a*H_s*W_s + y*W_s + x, the scales
 * concatenated in order.  term_mag (may be NULL) gets the sum of the
 * magnitudes of the terms of each output (for the relative tolerance). */
void oracle_detect_decode(const void* const* feats, int dt, const int* hw, const double* strides,
                          const double* anchors, int nscales, int na, int no, double* out,
                          double* term_mag) {
  int64_t row0 = 0;
  for (int s = 0; s < nscales; ++s) {
    int H = hw[2 * s], W = hw[2 * s + 1];
    for (int a = 0; a < na; ++a)
      for (int y = 0; y < H; ++y)
        for (int x = 0; x < W; ++x) {
          int64_t row = row0 + (int64_t)a * H * W + (int64_t)y * W + x;
          for (int k = 0; k < no; ++k) {
            int64_t src = ((int64_t)(a * no + k) * H + y) * W + x;
            double p = 1.0 / (1.0 + exp(-load_elem(feats[s], dt, src)));
            double o, m;
            if (k == 0) {
              o = (2.0 * p - 0.5 + x) * strides[s];
              m = (2.0 * p + 0.5 + x) * strides[s];
            } else if (k == 1) {
              o = (2.0 * p - 0.5 + y) * strides[s];
              m = (2.0 * p + 0.5 + y) * strides[s];
            } else if (k == 2) {
              o = (2.0 * p) * (2.0 * p) * anchors[(s * na + a) * 2 + 0];
              m = fabs(o);
            } else if (k == 3) {
              o = (2.0 * p) * (2.0 * p) * anchors[(s * na + a) * 2 + 1];
              m = fabs(o);
            } else {
              o = p;
              m = p;
            }
            out[row * no + k] = o;
            if (term_mag) term_mag[row * no + k] = m;
          }
        }
    row0 += (int64_t)na * H * W;
  }
}
