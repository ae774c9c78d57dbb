// chain.cpp -- op-chain IR, planner and CUDA code generator for fused
// elementwise chains, plus fuse_compile / fuse_launch.
//
// Method ("DeepJIT ... 串行小核墙"): section 4.1 fuses a chain of
// elementwise ops with several inputs into one kernel that reads each input
// once and writes once; section 4.2 vectorises the accesses (the pages use
// float4) with an alignment check that falls back to a scalar kernel and a
// tail handled outside the main loop; section 3.3 bakes the element count,
// vector width and tail switch into the source as constants.  ChannelShuffle
// ("算子与运行时", section 2) is fused as the gather index of input 0.
//
// GB300 design: 32-byte (ld/st .v8.b32) or 16-byte accesses per tensor per
// thread, several vectors in flight per thread, a grid of (SMs x resident
// CTAs) looping over whole chunks, and one CTA finishing the ragged remainder
// and the scalar tail after its share of the main loop.
#include <algorithm>
#include <atomic>
#include <cctype>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <sstream>
#include <thread>

#include "internal.h"

namespace fuse {

enum ChainOpCode {
  OP_ADD, OP_MUL, OP_SCALE, OP_RELU, OP_SIGMOID, OP_EXP, OP_CAST,
  OP_SIGMOID_FAST, OP_EXP_FAST  // "sigmoid:fast", "exp:fast": opt-in approximations
};

struct ChainOp {
  ChainOpCode op;
  float c = 0.f;             // scale constant
  fuse_dtype to = FUSE_F32;  // cast target
  int input = 0;             // add/mul operand
};

struct Chain {
  int groups = 0;  // ChannelShuffle groups on input 0 (0 = none)
  std::vector<ChainOp> ops;
  std::vector<fuse_dtype> in_dt;
  fuse_dtype out_dt = FUSE_F32;
};

constexpr int kMaxOps = 1024;
constexpr int kMaxInputs = 128;
constexpr int64_t kMaxElems = int64_t(1) << 40;

static std::string trim(const std::string& s) {
  size_t a = s.find_first_not_of(" \t\r\n"), b = s.find_last_not_of(" \t\r\n");
  return a == std::string::npos ? std::string() : s.substr(a, b - a + 1);
}

static int parse_dtype(const std::string& s, fuse_dtype* dt) {
  if (s == "f32") *dt = FUSE_F32;
  else if (s == "f16") *dt = FUSE_F16;
  else if (s == "bf16") *dt = FUSE_BF16;
  else return -1;
  return 0;
}

int parse_chain(const char* spec, fuse_dtype in_dt, Chain* out) {
  if (!spec) return fail(FUSE_E_NULL, "spec is NULL");
  if (!valid_dtype(in_dt)) return fail(FUSE_E_DTYPE, fmt("invalid input dtype %d", in_dt));
  Chain ch;
  ch.in_dt.push_back(in_dt);
  fuse_dtype cur = in_dt;
  std::stringstream ss(spec);
  std::string item;
  int pos = 0;
  while (std::getline(ss, item, ';')) {
    item = trim(item);
    if (item.empty()) continue;
    std::string name = item, arg;
    bool has_arg = false;
    if (size_t c = item.find(':'); c != std::string::npos) {
      name = trim(item.substr(0, c));
      arg = trim(item.substr(c + 1));
      has_arg = true;
    }
    if (name == "shuffle") {
      if (pos != 0) return fail(FUSE_E_SPEC, "shuffle must be the first item of the spec");
      char* end = nullptr;
      long g = has_arg ? strtol(arg.c_str(), &end, 10) : 0;
      if (!has_arg || arg.empty() || *end || g <= 0 || g > (1 << 20))
        return fail(FUSE_E_SPEC, fmt("bad shuffle groups '%s'", arg.c_str()));
      ch.groups = static_cast<int>(g);
      ++pos;
      continue;
    }
    ChainOp op{};
    if (name == "add" || name == "mul") {
      if (has_arg) return fail(FUSE_E_SPEC, fmt("'%s' takes no argument", name.c_str()));
      op.op = name == "add" ? OP_ADD : OP_MUL;
      op.input = static_cast<int>(ch.in_dt.size());
      ch.in_dt.push_back(cur);
    } else if (name == "scale") {
      char* end = nullptr;
      float c = has_arg ? strtof(arg.c_str(), &end) : 0.f;
      if (!has_arg || arg.empty() || *end || !std::isfinite(c))
        return fail(FUSE_E_SPEC, fmt("bad scale constant '%s'", arg.c_str()));
      op.op = OP_SCALE;
      op.c = c;
    } else if (name == "relu" || name == "sigmoid" || name == "exp") {
      // exp and sigmoid take the optional argument "fast": the hardware
      // approximation of 2^x on x * log2(e), per expression ("DeepJIT"
      // section 6.3: no global fast-math, intrinsics only where validated)
      const bool fast = has_arg && arg == "fast" && name != "relu";
      if (has_arg && !fast)
        return fail(FUSE_E_SPEC, fmt("'%s' takes no argument but 'fast' (exp, sigmoid)",
                                     name.c_str()));
      op.op = name == "relu" ? OP_RELU
              : name == "sigmoid" ? (fast ? OP_SIGMOID_FAST : OP_SIGMOID)
                                  : (fast ? OP_EXP_FAST : OP_EXP);
    } else if (name == "cast") {
      if (!has_arg || parse_dtype(arg, &op.to))
        return fail(FUSE_E_SPEC, fmt("bad cast target '%s' (f16, bf16 or f32)", arg.c_str()));
      op.op = OP_CAST;
      cur = op.to;
    } else {
      return fail(FUSE_E_SPEC, fmt("unknown op '%s'", item.c_str()));
    }
    ch.ops.push_back(op);
    ++pos;
    if (static_cast<int>(ch.ops.size()) > kMaxOps)
      return fail(FUSE_E_SPEC, fmt("more than %d ops", kMaxOps));
    if (static_cast<int>(ch.in_dt.size()) > kMaxInputs)
      return fail(FUSE_E_SPEC, fmt("more than %d input tensors", kMaxInputs));
  }
  ch.out_dt = cur;
  *out = std::move(ch);
  return FUSE_OK;
}

// ------------------------------------------------------------------ plan

struct ChainPlan {
  Chain ch;
  std::vector<int64_t> shape;
  int64_t n = 0;
  bool copy = false;  // no ops: bit copy of input 0
  int vec = 1;        // elements per vector
  int block = 256;
  int unroll = 1;
  bool vec_ok = false;
  int64_t C = 1, HW = 1;
  bool dynamic = false;  // shape bucket: the leading dimension comes with the launch
  bool debug = false;    // FUSE_DEBUG_BOUNDS: every index checked against its tensor
  bool prefetch = false;  // L2 prefetch of the first chunk before the launch-order wait
  bool pack2 = false;     // adds and multiplies as packed fp32 pairs (f32x2)
  int64_t inner = 1;     // elements per unit of the leading dimension
  std::string source;
};

static int env_int(const char* name, int dflt) {
  const char* e = getenv(name);
  return e && *e ? atoi(e) : dflt;
}

int plan_chain(const char* spec, const int64_t* shape, int ndim, fuse_dtype in_dt, ChainPlan* p) {
  if (int rc = parse_chain(spec, in_dt, &p->ch)) return rc;
  if (!shape && ndim > 0) return fail(FUSE_E_NULL, "shape is NULL");
  if (ndim < 1 || ndim > 8) return fail(FUSE_E_SHAPE, fmt("ndim %d outside 1..8", ndim));
  int64_t n = 1;
  for (int i = 0; i < ndim; ++i) {
    if (shape[i] < 0) return fail(FUSE_E_SHAPE, fmt("negative dimension %lld", (long long)shape[i]));
    if (shape[i] && n > kMaxElems / shape[i])
      return fail(FUSE_E_SHAPE, "more than 2^40 elements");
    n *= shape[i];
    p->shape.push_back(shape[i]);
  }
  if (n > kMaxElems) return fail(FUSE_E_SHAPE, "more than 2^40 elements");
  p->n = n;
  p->inner = 1;
  for (int i = 1; i < ndim; ++i) p->inner *= shape[i];
  const Chain& ch = p->ch;
  if (ch.groups) {
    if (ndim != 4) return fail(FUSE_E_SHAPE, "shuffle needs a 4-D NCHW shape");
    if (shape[1] % ch.groups)
      return fail(FUSE_E_SHAPE, fmt("channels %lld not divisible by %d groups",
                                    (long long)shape[1], ch.groups));
    p->C = shape[1];
    p->HW = shape[2] * shape[3];
  }
  p->copy = ch.ops.empty();
  // Elements per vector: the widest access (32, 16, 8 or 4 bytes of the
  // narrowest tensor) whose register words -- every input's and the
  // output's share of one vector -- fit the budget, so that chains with many
  // inputs keep enough warps resident.
  int minb = dtype_bytes(ch.out_dt), bytes_per_elem = dtype_bytes(ch.out_dt);
  for (auto d : ch.in_dt) {
    minb = std::min(minb, dtype_bytes(d));
    bytes_per_elem += dtype_bytes(d);
  }
  bool transcendental = false;
  for (auto& op : ch.ops)
    transcendental = transcendental || op.op == OP_EXP || op.op == OP_SIGMOID ||
                     op.op == OP_EXP_FAST || op.op == OP_SIGMOID_FAST;
  // Measured on GB300 (sweep over the chain workloads): chains touching 12 or
  // more tensors run fastest with a small per-thread footprint (more warps,
  // the 13-input chain 1.64 ms vs 1.86 ms), others with the widest vectors
  // (the 6-tensor chain 537 us vs 558 us); chains with exp/sigmoid lose by
  // unrolling (more registers, fewer warps to hide the arithmetic).
  const int tensors = static_cast<int>(ch.in_dt.size()) + 1;
  const int budget = env_int("FUSE_CHAIN_WORD_BUDGET", tensors >= 12 ? 32 : 64);
  int vec_bytes = env_int("FUSE_CHAIN_VEC_BYTES", 32);
  if (vec_bytes != 4 && vec_bytes != 8 && vec_bytes != 16 && vec_bytes != 32) vec_bytes = 32;
  while (vec_bytes > 4 && (vec_bytes / minb) * bytes_per_elem / 4 > budget) vec_bytes /= 2;
  p->vec = vec_bytes / minb;
  const int words = p->vec * bytes_per_elem / 4;
  // vectors in flight per thread: enough to cover latency, bounded registers
  int max_unroll = env_int("FUSE_CHAIN_UNROLL", transcendental ? 1 : 2);
  p->unroll = 1;
  while (p->unroll * 2 <= max_unroll && words * p->unroll * 2 <= budget) p->unroll *= 2;
  p->block = env_int("FUSE_CHAIN_BLOCK", 256);
  if (p->block < 32 || p->block > 1024 || p->block % 32) p->block = 256;
  // Small tensors: shrink the chunk (fewer vectors in flight per thread, then
  // smaller CTAs, then 16-byte vectors) until there are about 8 CTAs per SM,
  // so that every SM has loads in flight.
  const int64_t want_ctas = int64_t(8) * default_sms();
  auto chunks = [&]() { return n / p->vec / (int64_t(p->block) * p->unroll); };
  while (chunks() < want_ctas) {
    if (p->unroll > 1) p->unroll /= 2;
    else if (p->block > 128) p->block /= 2;
    else if (p->vec * minb > 16) p->vec /= 2;
    else break;
  }
  p->vec_ok = !ch.groups || (p->HW % p->vec == 0);
  p->debug = env_int("FUSE_DEBUG_BOUNDS", 0) == 1;
  // the bulk prefetch needs 16-byte aligned ranges: every tensor's vector a
  // multiple of 16 bytes (the vector kernel's pointers are 16-byte aligned)
  p->prefetch = env_int("FUSE_CHAIN_PREFETCH", 1) == 1 && p->vec * minb >= 16;
  // two elements a step, the adds and multiplies of add / mul / scale and of
  // the fast forms as one packed instruction each (FUSE_CHAIN_F32X2=0 turns
  // it off).  The accurate sigmoid stays per element: pairing its add made
  // the 16-op shuffle chain slower (64.0 against 61.6 us on GB300).
  bool arith = false;
  for (auto& op : p->ch.ops)
    arith = arith || op.op == OP_ADD || op.op == OP_MUL || op.op == OP_SCALE ||
            op.op == OP_EXP_FAST || op.op == OP_SIGMOID_FAST;
  p->pack2 = env_int("FUSE_CHAIN_F32X2", 1) == 1 && p->vec % 2 == 0 && arith;
  return FUSE_OK;
}

// ------------------------------------------------------------------ codegen

// elem_of_input: expression of an operand element, with "@" standing for the
// input number
static std::string operand(const std::string& elem_of_input, int input) {
  std::string out;
  for (char c : elem_of_input) out += c == '@' ? std::to_string(input) : std::string(1, c);
  return out;
}

static void emit_op(std::ostringstream& s, const ChainOp& op, const std::string& elem_of_input) {
  switch (op.op) {
    case OP_ADD: s << "      x = x + " << operand(elem_of_input, op.input) << ";\n"; break;
    case OP_MUL: s << "      x = x * " << operand(elem_of_input, op.input) << ";\n"; break;
    case OP_SCALE: s << "      x = x * " << hex_float(op.c) << ";\n"; break;
    case OP_RELU: s << "      x = x > 0.f ? x : 0.f;\n"; break;
    // 1 / (1 + exp(-x)); the reciprocal of the value >= 1 by the hardware
    // approximation, documented to within 1 ulp (common.cuh), in place of the
    // IEEE division
    case OP_SIGMOID: s << "      x = sigmoid(x);\n"; break;
    case OP_EXP: s << "      x = expf(x);\n"; break;
    case OP_SIGMOID_FAST: s << "      x = sigmoid_fast(x);\n"; break;
    case OP_EXP_FAST: s << "      x = exp_fast(x);\n"; break;
    case OP_CAST:
      if (op.to == FUSE_F16) s << "      x = round_f16(x);\n";
      else if (op.to == FUSE_BF16) s << "      x = round_bf16(x);\n";
      else s << "      /* cast:f32 keeps the fp32 value */\n";
      break;
  }
}

// the same op on a pair of elements x0, x1 (operands elem0 / elem1)
static void emit_op2(std::ostringstream& s, const ChainOp& op, const std::string& elem0,
                     const std::string& elem1) {
  switch (op.op) {
    case OP_ADD:
      s << "      add2(x0, x1, " << operand(elem0, op.input) << ", " << operand(elem1, op.input)
        << ");\n";
      break;
    case OP_MUL:
      s << "      mul2(x0, x1, " << operand(elem0, op.input) << ", " << operand(elem1, op.input)
        << ");\n";
      break;
    case OP_SCALE:
      s << "      mul2(x0, x1, " << hex_float(op.c) << ", " << hex_float(op.c) << ");\n";
      break;
    case OP_EXP_FAST: s << "      exp_fast2(x0, x1);\n"; break;
    case OP_SIGMOID_FAST: s << "      sigmoid_fast2(x0, x1);\n"; break;
    default: {
      std::ostringstream one;
      emit_op(one, op, elem0);
      std::string t = one.str(), a, b;
      for (size_t i = 0; i < t.size(); ++i) {
        // the scalar statement on x, once for each element of the pair
        const bool var = t[i] == 'x' && (i == 0 || !isalnum(static_cast<unsigned char>(t[i - 1])) &&
                                                      t[i - 1] != '_') &&
                         (i + 1 == t.size() || !isalnum(static_cast<unsigned char>(t[i + 1])) &&
                                                   t[i + 1] != '_');
        a += var ? std::string("x0") : std::string(1, t[i]);
        b += var ? std::string("x1") : std::string(1, t[i]);
      }
      s << a << b;
    }
  }
}

static std::string gen_chain_source(const ChainPlan& p, const char* spec) {
  const Chain& ch = p.ch;
  const int nin = static_cast<int>(ch.in_dt.size());
  const bool small = p.n < (int64_t(1) << 31);
  std::ostringstream s;
  s << "// fused chain: " << spec << "\n";
  s << "#include \"fuse/common.cuh\"\n";
  s << "typedef " << (small ? "unsigned" : "long long") << " idx_t;\n";
  s << "constexpr long long N = " << p.n << "LL;\n";
  s << "constexpr int VEC = " << p.vec << ";\n";
  s << "constexpr int BLOCK = " << p.block << ";\n";
  s << "constexpr int UNROLL = " << p.unroll << ";\n";
  s << "constexpr long long NVEC = N / VEC;\n";
  s << "constexpr long long CHUNK = (long long)BLOCK * UNROLL;\n";
  s << "constexpr long long NFULL = NVEC / CHUNK;\n";
  s << "constexpr int NREM = (int)(NVEC - NFULL * CHUNK);\n";
  s << "constexpr int TAIL = (int)(N - NVEC * VEC);\n";
  s << "constexpr int NIN = " << nin << ";\n";
  for (int j = 0; j < nin; ++j) {
    s << "constexpr int DT" << j << " = " << ch.in_dt[j] << ";  // " << dtype_name(ch.in_dt[j])
      << "\n";
    s << "constexpr int NW" << j << " = VEC * Dt<DT" << j << ">::bytes / 4;\n";
  }
  s << "constexpr int DTO = " << ch.out_dt << ";  // " << dtype_name(ch.out_dt) << "\n";
  s << "constexpr int NWO = VEC * Dt<DTO>::bytes / 4;\n";
  if (p.debug) {
    // debug bounds checks: the launch always passes the element count and
    // the device error word; an index outside its tensor records code 3
    // there and the access is skipped
    s << "struct Args { const void* in[NIN]; void* out; long long n; int* err; };\n";
    s << (p.dynamic ? "#define SIZE_N(a) ((a).n)\n" : "#define SIZE_N(a) N\n");
    s << "__device__ __forceinline__ bool in_bounds(const Args& a, long long i, long long lim) {\n"
         "  if (i >= 0 && i < lim) return true;\n"
         "  atomicExch(a.err, 3);\n"
         "  return false;\n"
         "}\n\n";
  } else if (p.dynamic) {
    // shape bucket: N above is the largest element count; the launch passes
    // the actual one
    s << "struct Args { const void* in[NIN]; void* out; long long n; };\n";
    s << "#define SIZE_N(a) ((a).n)\n\n";
  } else {
    s << "struct Args { const void* in[NIN]; void* out; };\n";
    s << "#define SIZE_N(a) N\n\n";
  }

  // index of input 0 for an output element / vector (ChannelShuffle prologue)
  if (ch.groups) {
    s << "// ChannelShuffle: output channel j*G + i reads input channel i*(C/G) + j\n";
    s << "constexpr idx_t C = " << p.C << ", HW = " << p.HW << ", G = " << ch.groups
      << ", CPG = C / G;\n";
    s << "__device__ __forceinline__ idx_t src_elem(idx_t e) {\n"
         "  const idx_t plane = e / HW, off = e - plane * HW;\n"
         "  const idx_t nn = plane / C, co = plane - nn * C;\n"
         "  const idx_t ci = (co % G) * CPG + co / G;\n"
         "  return (nn * C + ci) * HW + off;\n"
         "}\n";
    if (p.vec_ok) {
      s << "constexpr idx_t VPP = HW / VEC;  // vectors per plane\n";
      s << "__device__ __forceinline__ idx_t src_vec(idx_t v) {\n"
           "  const idx_t plane = v / VPP, off = v - plane * VPP;\n"
           "  const idx_t nn = plane / C, co = plane - nn * C;\n"
           "  const idx_t ci = (co % G) * CPG + co / G;\n"
           "  return (nn * C + ci) * VPP + off;\n"
           "}\n";
    }
  } else {
    s << "__device__ __forceinline__ idx_t src_elem(idx_t e) { return e; }\n";
    s << "__device__ __forceinline__ idx_t src_vec(idx_t v) { return v; }\n";
  }

  // per-element chain on register vectors
  s << "\n// the chain, one element at a time, in fp32 registers\n";
  s << "__device__ __forceinline__ void apply(";
  for (int j = 0; j < nin; ++j) s << "const u32 (&w" << j << ")[NW" << j << "], ";
  s << "u32 (&wo)[NWO]) {\n";
  if (p.copy) {
    s << "  static_assert(NWO == NW0, \"copy\");\n"
         "#pragma unroll\n  for (int i = 0; i < NWO; ++i) wo[i] = w0[i];\n}\n";
  } else if (p.pack2) {
    s << "  float y[VEC];\n#pragma unroll\n  for (int e = 0; e < VEC; e += 2) {\n";
    s << "      float x0 = get_elem<DT0>(w0, e), x1 = get_elem<DT0>(w0, e + 1);\n";
    for (auto& op : ch.ops) emit_op2(s, op, "get_elem<DT@>(w@, e)", "get_elem<DT@>(w@, e + 1)");
    s << "      y[e] = x0;\n      y[e + 1] = x1;\n  }\n  pack_vec<DTO>(y, wo);\n}\n";
  } else {
    s << "  float y[VEC];\n#pragma unroll\n  for (int e = 0; e < VEC; ++e) {\n";
    s << "      float x = get_elem<DT0>(w0, e);\n";
    for (auto& op : ch.ops) emit_op(s, op, "get_elem<DT@>(w@, e)");
    s << "      y[e] = x;\n  }\n  pack_vec<DTO>(y, wo);\n}\n";
  }

  // scalar chain for one element (tail and fallback kernel)
  s << "\n__device__ __forceinline__ void apply_elem(const Args& a, idx_t e) {\n";
  if (p.debug)  // every access below is at e (inputs 1.., output) or src_elem(e) (input 0)
    s << "  if (!in_bounds(a, e, SIZE_N(a)) || !in_bounds(a, src_elem(e), SIZE_N(a))) return;\n";
  if (p.copy) {
    s << "  static_cast<typename Dt<DTO>::storage*>(a.out)[e] =\n"
         "      static_cast<const typename Dt<DT0>::storage*>(a.in[0])[src_elem(e)];\n}\n";
  } else {
    s << "  float x = load_elem<DT0>(a.in[0], src_elem(e));\n";
    for (auto& op : ch.ops) emit_op(s, op, "load_elem<DT@>(a.in[@], e)");
    s << "  store_elem<DTO>(a.out, e, x);\n}\n";
  }

  // vector kernel
  if (p.vec_ok) {
    s << "\n// vectors [v0, v0 + UNROLL*BLOCK) with stride BLOCK; CHECK: bound by nvec\n";
    s << "template <bool CHECK>\n__device__ __forceinline__ void do_chunk(const Args& a, idx_t v0, "
         "idx_t nvec) {\n";
    for (int j = 0; j < nin; ++j) s << "  u32 r" << j << "[UNROLL][NW" << j << "];\n";
    // debug: a vector whose index or source index falls outside the
    // tensors is neither loaded nor stored
    const char* dbg = p.debug ? "    if (!in_bounds(a, v, nvec) || !in_bounds(a, src_vec(v), nvec)) continue;\n"
                              : "";
    s << "#pragma unroll\n  for (int u = 0; u < UNROLL; ++u) {\n"
         "    const idx_t v = v0 + (idx_t)u * BLOCK;\n"
         "    if (CHECK && v >= nvec) break;\n" << dbg;
    for (int j = 0; j < nin; ++j) {
      s << "    load_words(static_cast<const u32*>(a.in[" << j << "]) + (idx_t)"
        << (j == 0 ? "src_vec(v)" : "v") << " * NW" << j << ", r" << j << "[u]);\n";
    }
    s << "  }\n#pragma unroll\n  for (int u = 0; u < UNROLL; ++u) {\n"
         "    const idx_t v = v0 + (idx_t)u * BLOCK;\n"
         "    if (CHECK && v >= nvec) break;\n" << dbg <<
         "    u32 wo[NWO];\n    apply(";
    for (int j = 0; j < nin; ++j) s << "r" << j << "[u], ";
    s << "wo);\n    store_words(static_cast<u32*>(a.out) + v * NWO, wo);\n  }\n}\n";
    if (p.prefetch) {
      // Before the wait for the previous kernel on the stream (programmatic
      // dependent launch lets this grid's first CTAs start while it drains):
      // one thread per CTA asks L2 for the CTA's first chunk of every input.
      // L2 is where global memory is coherent, so a line the previous kernel
      // still writes is updated there, and every load of the chunk is issued
      // after the wait.
      s << "\n__device__ __forceinline__ void prefetch_chunk(const Args& a, idx_t c) {\n";
      for (int j = 0; j < nin; ++j) {
        if (j == 0 && ch.groups) {
          // the shuffled input: the chunk's source is one run per plane
          s << "  for (idx_t v = c * (idx_t)CHUNK, e = v + (idx_t)CHUNK; v < e;) {\n"
               "    const idx_t pe = (v / VPP + 1) * VPP, se = pe < e ? pe : e;\n"
               "    prefetch_l2(static_cast<const u32*>(a.in[0]) + (idx_t)src_vec(v) * NW0,\n"
               "                (unsigned)((se - v) * NW0 * 4));\n"
               "    v = se;\n  }\n";
        } else {
          s << "  prefetch_l2(static_cast<const u32*>(a.in[" << j << "]) + c * (idx_t)CHUNK * NW" << j
            << ", (unsigned)(CHUNK * NW" << j << " * 4));\n";
        }
      }
      s << "}\n";
    }
    // sizes: compile-time constants for a fixed shape (the compiler folds
    // every branch below), the launch's element count for a shape bucket
    s << "\nextern \"C\" __global__ void __launch_bounds__(BLOCK) fuse_chain_vec(const Args a) {\n";
    if (p.prefetch)
      s << "  if (threadIdx.x == 0 && (idx_t)blockIdx.x < (idx_t)SIZE_N(a) / VEC / (idx_t)CHUNK)\n"
           "    prefetch_chunk(a, blockIdx.x);\n";
    s << "  pdl_enter();\n"
         "  const idx_t n = (idx_t)SIZE_N(a), nvec = n / VEC, nfull = nvec / (idx_t)CHUNK;\n"
         "  const idx_t nrem = nvec - nfull * (idx_t)CHUNK, tail = n - nvec * VEC;\n"
         "  for (idx_t c = blockIdx.x; c < nfull; c += gridDim.x)\n"
         "    do_chunk<false>(a, c * (idx_t)CHUNK + threadIdx.x, nvec);\n"
         "  if (nrem > 0 || tail > 0) {\n"
         "    // the CTA with the fewest full chunks takes the remainder and the tail\n"
         "    if (blockIdx.x == (unsigned)(nfull % gridDim.x)) {\n"
         "      if (nrem > 0) do_chunk<true>(a, nfull * (idx_t)CHUNK + threadIdx.x, nvec);\n"
         "      if (threadIdx.x < tail) apply_elem(a, nvec * VEC + threadIdx.x);\n"
         "    }\n  }\n}\n";
  }
  // scalar kernel: any alignment
  s << "\nextern \"C\" __global__ void __launch_bounds__(256) fuse_chain_scalar(const Args a) {\n"
         "  pdl_enter();\n"
       "  const idx_t n = (idx_t)SIZE_N(a);\n"
       "  for (idx_t e = (idx_t)blockIdx.x * 256 + threadIdx.x; e < n;"
       " e += (idx_t)gridDim.x * 256)\n"
       "    apply_elem(a, e);\n}\n";
  return s.str();
}

// ------------------------------------------------------------------ handle

}  // namespace fuse

struct fuse_chain {
  fuse::ChainPlan plan;
  std::shared_ptr<fuse::Module> mod;
  std::mutex mu;
  struct PerDevice {
    int device, sms;
    CUfunction vec_fn, scalar_fn;
    int occ_vec, occ_scalar;  // resident CTAs per SM of each kernel
  };
  // one entry per device that launched the chain; entries never move (a
  // launch keeps using its entry after the lock is released)
  std::vector<std::unique_ptr<PerDevice>> dev;
};

namespace fuse {

static int chain_device_state(fuse_chain* h, const DeviceInfo& d, fuse_chain::PerDevice** out) {
  std::lock_guard<std::mutex> lk(h->mu);
  for (auto& pd : h->dev)
    if (pd->device == d.ordinal) {
      *out = pd.get();
      return FUSE_OK;
    }
  fuse_chain::PerDevice pd{};
  pd.device = d.ordinal;
  pd.sms = d.sms;
  const DriverApi* api;
  if (int rc = driver(&api)) return rc;
  const ChainPlan& p = h->plan;
  if (int rc = jit_function(*h->mod, "fuse_chain_scalar", d, &pd.scalar_fn)) return rc;
  CUresult r = api->OccupancyMaxActiveBlocksPerMultiprocessor(&pd.occ_scalar, pd.scalar_fn, 256, 0);
  if (r != CUDA_SUCCESS) return cuda_fail(r, "cuOccupancyMaxActiveBlocksPerMultiprocessor");
  if (p.vec_ok) {
    if (int rc = jit_function(*h->mod, "fuse_chain_vec", d, &pd.vec_fn)) return rc;
    r = api->OccupancyMaxActiveBlocksPerMultiprocessor(&pd.occ_vec, pd.vec_fn, p.block, 0);
    if (r != CUDA_SUCCESS) return cuda_fail(r, "cuOccupancyMaxActiveBlocksPerMultiprocessor");
  }
  h->dev.push_back(std::make_unique<fuse_chain::PerDevice>(pd));
  *out = h->dev.back().get();
  return FUSE_OK;
}

// Grids for n elements.  Vector kernel: one chunk per CTA, so the block
// scheduler hands chunks to SMs as they free up and the last wave is at most
// one chunk long (FUSE_CHAIN_CTAS_PER_SM instead sizes a persistent grid of
// SMs x that many CTAs).  Scalar kernel: a grid-stride loop over resident CTAs.
static void chain_grids(const ChainPlan& p, const fuse_chain::PerDevice& pd, int64_t n,
                        unsigned* vec_grid, unsigned* scalar_grid) {
  const int64_t want = (n + 255) / 256;
  *scalar_grid = static_cast<unsigned>(std::max<int64_t>(
      1, std::min<int64_t>(want, int64_t(pd.sms) * std::max(pd.occ_scalar, 1))));
  static const int per_sm = env_int("FUSE_CHAIN_CTAS_PER_SM", 0);  // read once
  const int64_t nfull = (n / p.vec) / (int64_t(p.block) * p.unroll);
  int64_t cap = int64_t(1) << 30;
  if (per_sm > 0) cap = int64_t(pd.sms) * std::min(per_sm, std::max(pd.occ_vec, 1));
  *vec_grid = static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(nfull, cap)));
}

int chain_compile(const char* spec, const int64_t* shape, int ndim, fuse_dtype in_dt,
                  fuse_chain** out, bool bucket) {
  auto h = std::make_unique<fuse_chain>();
  if (int rc = plan_chain(spec, shape, ndim, in_dt, &h->plan)) return rc;
  h->plan.dynamic = bucket;
  h->plan.source = gen_chain_source(h->plan, spec);
  if (int rc = jit_compile(h->plan.source, "fuse_chain", &h->mod)) return rc;
  // load now when a device is present, so that the first launch does no work
  DeviceInfo d;
  fuse_chain::PerDevice* pd;
  if (current_device(&d) == FUSE_OK) {
    if (int rc = chain_device_state(h.get(), d, &pd)) return rc;
  }
  clear_error();
  *out = h.release();
  return FUSE_OK;
}

int chain_source(const char* spec, const int64_t* shape, int ndim, fuse_dtype in_dt,
                 std::string* src, bool bucket) {
  ChainPlan p;
  if (int rc = plan_chain(spec, shape, ndim, in_dt, &p)) return rc;
  p.dynamic = bucket;
  *src = gen_chain_source(p, spec);
  return FUSE_OK;
}

// rows < 0: the compiled leading dimension.  A bucket handle accepts any
// 0 <= rows <= its leading dimension; a fixed handle only its own.
int chain_launch(fuse_chain* h, const void* const* inputs, int n_in, void* output, void* stream,
                 int64_t rows) {
  const ChainPlan& p = h->plan;
  const int nin = static_cast<int>(p.ch.in_dt.size());
  if (n_in != nin) return fail(FUSE_E_ARG, fmt("chain takes %d inputs, got %d", nin, n_in));
  int64_t n = p.n;
  if (rows >= 0) {
    if (rows > p.shape[0] || (!p.dynamic && rows != p.shape[0]))
      return fail(FUSE_E_SHAPE,
                  fmt("leading dimension %lld: the handle was compiled for %s%lld",
                      (long long)rows, p.dynamic ? "at most " : "", (long long)p.shape[0]));
    n = rows * p.inner;
  }
  if (n == 0) return FUSE_OK;
  if (!inputs) return fail(FUSE_E_NULL, "inputs is NULL");
  if (!output) return fail(FUSE_E_NULL, "output is NULL");
  bool aligned = aligned16(output);
  for (int j = 0; j < nin; ++j) {
    if (!inputs[j]) return fail(FUSE_E_NULL, fmt("input %d is NULL", j));
    aligned = aligned && aligned16(inputs[j]);
  }
  if (p.ch.groups && output == inputs[0])
    return fail(FUSE_E_ARG, "a shuffled chain cannot write over its input 0");
  DeviceInfo d;
  if (int rc = current_device(&d)) return rc;
  fuse_chain::PerDevice* pd;
  if (int rc = chain_device_state(h, d, &pd)) return rc;
  // kernel parameter: the Args struct {in[NIN], out[, n][, err]} as 8-byte
  // words (the debug build always has n, then the device error word)
  uint64_t args[kMaxInputs + 3];  // on the stack: no allocation per launch
  for (int j = 0; j < nin; ++j) args[j] = reinterpret_cast<uintptr_t>(inputs[j]);
  args[nin] = reinterpret_cast<uintptr_t>(output);
  args[nin + 1] = static_cast<uint64_t>(n);
  if (p.debug) {
    CUdeviceptr err;
    if (int rc = device_error_word(d.ordinal, &err)) return rc;
    args[nin + 2] = static_cast<uint64_t>(err);
  }
  void* kargs[] = {args};
  unsigned vec_grid, scalar_grid;
  chain_grids(p, *pd, n, &vec_grid, &scalar_grid);
  // 32-byte accesses need 32-byte alignment when a vector spans 32 bytes
  bool use_vec = p.vec_ok && aligned;
  if (use_vec) {
    for (int j = 0; j <= nin; ++j) {
      const void* ptr = j < nin ? inputs[j] : output;
      fuse_dtype dt = j < nin ? p.ch.in_dt[j] : p.ch.out_dt;
      int bytes = p.vec * dtype_bytes(dt);
      int need = bytes >= 32 ? 32 : bytes;
      if (reinterpret_cast<uintptr_t>(ptr) % need) use_vec = false;
    }
  }
  if (use_vec) return launch(pd->vec_fn, vec_grid, p.block, 0, stream, kargs);
  return launch(pd->scalar_fn, scalar_grid, 256, 0, stream, kargs);
}

}  // namespace fuse

// ------------------------------------------------------------------ C ABI

static int copy_source(const std::string& src, char* buf, size_t cap, size_t* len) {
  if (len) *len = src.size();
  if (buf && cap) {
    size_t n = std::min(cap - 1, src.size());
    memcpy(buf, src.data(), n);
    buf[n] = '\0';
  }
  return FUSE_OK;
}

extern "C" {

int fuse_compile(const char* spec, const int64_t* shape, int ndim, fuse_dtype in_dtype,
                 fuse_handle* out) {
  fuse::NvtxRange nvtx_range("fuse_compile");
  if (!out) return fuse::fail(FUSE_E_NULL, "out is NULL");
  *out = nullptr;
  return fuse::chain_compile(spec, shape, ndim, in_dtype, out, false);
}

int fuse_compile_bucket(const char* spec, const int64_t* shape, int ndim, fuse_dtype in_dtype,
                        fuse_handle* out) {
  fuse::NvtxRange nvtx_range("fuse_compile_bucket");
  if (!out) return fuse::fail(FUSE_E_NULL, "out is NULL");
  *out = nullptr;
  return fuse::chain_compile(spec, shape, ndim, in_dtype, out, true);
}

int fuse_warmup(const char* list, int threads, int* compiled, int* cached) {
  fuse::NvtxRange nvtx_range("fuse_warmup");
  using namespace fuse;
  if (compiled) *compiled = 0;
  if (cached) *cached = 0;
  if (!list) return fail(FUSE_E_NULL, "list is NULL");
  auto trim = [](std::string t) {
    const size_t a = t.find_first_not_of(" \t\r"), b = t.find_last_not_of(" \t\r");
    return a == std::string::npos ? std::string() : t.substr(a, b - a + 1);
  };
  // every line: spec | d0,d1,... | dtype [| bucket]; its kernel source
  struct Entry {
    int line;
    std::string source;
  };
  std::vector<Entry> entries;
  std::istringstream in(list);
  std::string text;
  for (int ln = 1; std::getline(in, text); ++ln) {
    text = trim(text);
    if (text.empty() || text[0] == '#') continue;
    std::vector<std::string> f;
    for (size_t a = 0;;) {
      const size_t b = text.find('|', a);
      f.push_back(trim(text.substr(a, b == std::string::npos ? std::string::npos : b - a)));
      if (b == std::string::npos) break;
      a = b + 1;
    }
    if (f.size() < 3 || f.size() > 4 || (f.size() == 4 && f[3] != "bucket"))
      return fail(FUSE_E_SPEC,
                  fmt("warm-up list line %d: want 'spec | d0,d1,... | f32|f16|bf16 [| bucket]'", ln));
    std::vector<int64_t> shape;
    for (size_t a = 0;;) {
      const size_t b = f[1].find(',', a);
      const std::string d = trim(f[1].substr(a, b == std::string::npos ? std::string::npos : b - a));
      char* end = nullptr;
      const long long v = strtoll(d.c_str(), &end, 10);
      if (d.empty() || *end || v < 0)
        return fail(FUSE_E_SHAPE, fmt("warm-up list line %d: bad dimension '%s'", ln, d.c_str()));
      shape.push_back(v);
      if (b == std::string::npos) break;
      a = b + 1;
    }
    const fuse_dtype dt = f[2] == "f32" ? FUSE_F32 : f[2] == "f16" ? FUSE_F16 : FUSE_BF16;
    if (f[2] != "f32" && f[2] != "f16" && f[2] != "bf16")
      return fail(FUSE_E_DTYPE, fmt("warm-up list line %d: dtype '%s'", ln, f[2].c_str()));
    ChainPlan p;
    if (int rc = plan_chain(f[0].c_str(), shape.data(), static_cast<int>(shape.size()), dt, &p))
      return fail(rc, fmt("warm-up list line %d: %s", ln, last_error_cstr()));
    p.dynamic = f.size() == 4;
    entries.push_back({ln, gen_chain_source(p, f[0].c_str())});
  }
  // compile on worker threads (distinct sources compile in parallel); the
  // first error, with its line, is reported on the calling thread
  const int n = static_cast<int>(entries.size());
  int nt = threads > 0 ? threads : static_cast<int>(std::thread::hardware_concurrency());
  nt = std::max(1, std::min({nt, 16, n}));
  std::atomic<int> next{0}, n_compiled{0}, n_cached{0};
  std::mutex err_mu;
  int err_rc = FUSE_OK;
  std::string err_msg;
  auto work = [&] {
    for (int i; (i = next.fetch_add(1)) < n;) {
      {
        std::lock_guard<std::mutex> lk(err_mu);
        if (err_rc != FUSE_OK) return;
      }
      std::shared_ptr<Module> m;
      bool fresh = false;
      if (int rc = jit_compile(entries[i].source, "fuse_chain", &m, &fresh)) {
        std::lock_guard<std::mutex> lk(err_mu);
        if (err_rc == FUSE_OK) {
          err_rc = rc;
          err_msg = fmt("warm-up list line %d: ", entries[i].line) + last_error_cstr();
        }
        return;
      }
      (fresh ? n_compiled : n_cached).fetch_add(1);
    }
  };
  std::vector<std::thread> pool;
  for (int t = 1; t < nt; ++t) pool.emplace_back(work);
  work();
  for (auto& t : pool) t.join();
  if (err_rc != FUSE_OK) return fail(err_rc, err_msg);
  if (compiled) *compiled = n_compiled.load();
  if (cached) *cached = n_cached.load();
  clear_error();
  return FUSE_OK;
}

int fuse_bucket(int64_t n, int64_t* bucket) {
  if (!bucket) return fuse::fail(FUSE_E_NULL, "bucket is NULL");
  if (n < 0 || n > (int64_t(1) << 40)) return fuse::fail(FUSE_E_SHAPE, "n outside 0..2^40");
  int64_t b = 1;
  while (b < n) b <<= 1;
  *bucket = b;
  return FUSE_OK;
}

int fuse_num_inputs(fuse_handle h, int* n_in, fuse_dtype* out_dtype) {
  if (!h) return fuse::fail(FUSE_E_ARG, "NULL handle");
  if (n_in) *n_in = static_cast<int>(h->plan.ch.in_dt.size());
  if (out_dtype) *out_dtype = h->plan.ch.out_dt;
  return FUSE_OK;
}

int fuse_input_dtypes(fuse_handle h, fuse_dtype* dts, int cap) {
  if (!h) return fuse::fail(FUSE_E_ARG, "NULL handle");
  if (!dts) return fuse::fail(FUSE_E_NULL, "dts is NULL");
  int n = static_cast<int>(h->plan.ch.in_dt.size());
  if (cap < n) return fuse::fail(FUSE_E_ARG, fuse::fmt("need room for %d dtypes", n));
  for (int i = 0; i < n; ++i) dts[i] = h->plan.ch.in_dt[i];
  return FUSE_OK;
}

int fuse_launch(fuse_handle h, const void* const* inputs, int n_in, void* output, void* stream) {
  fuse::NvtxRange nvtx_range("fuse_launch");
  if (!h) return fuse::fail(FUSE_E_ARG, "NULL handle");
  return fuse::chain_launch(h, inputs, n_in, output, stream, -1);
}

int fuse_launch_rows(fuse_handle h, const void* const* inputs, int n_in, void* output,
                     int64_t rows, void* stream) {
  fuse::NvtxRange nvtx_range("fuse_launch_rows");
  if (!h) return fuse::fail(FUSE_E_ARG, "NULL handle");
  if (rows < 0) return fuse::fail(FUSE_E_SHAPE, "rows < 0");
  return fuse::chain_launch(h, inputs, n_in, output, stream, rows);
}

int fuse_release(fuse_handle h) {
  delete h;  // the compiled module stays in the cache for the life of the process
  return FUSE_OK;
}

int fuse_source(const char* spec, const int64_t* shape, int ndim, fuse_dtype in_dtype, char* buf,
                size_t cap, size_t* len) {
  std::string src;
  if (int rc = fuse::chain_source(spec, shape, ndim, in_dtype, &src, false)) return rc;
  return copy_source(src, buf, cap, len);
}

int fuse_source_bucket(const char* spec, const int64_t* shape, int ndim, fuse_dtype in_dtype,
                       char* buf, size_t cap, size_t* len) {
  std::string src;
  if (int rc = fuse::chain_source(spec, shape, ndim, in_dtype, &src, true)) return rc;
  return copy_source(src, buf, cap, len);
}

}  // extern "C"
