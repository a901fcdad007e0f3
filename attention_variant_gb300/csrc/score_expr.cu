// score_expr.cu -- score_mod expressions compiled into the fused kernel at
// run time.
//
// The Flashlight pages' central point is that an attention variant written as
// a plain elementwise expression over the score and its indices is fused into
// the same single-pass kernel as the built-in variants, with no per-variant
// template written by hand (talk notes, "Compiler design" 1-4 and the
// comparison with FlexAttention's score_mod/mask_mod interface; gist.science
// summary, "Methodology").  Here the expression is a string in a small grammar
// (fl_attn.h, FL_MOD_EXPR).  The library
//   1. parses it and writes the equivalent fp32 CUDA expression
//      (score_expr_translate): numbers become float literals, names map to
//      fixed helper functions, anything outside the grammar is refused, so
//      what is compiled is exactly what the grammar means;
//   2. on the first use of an expression on a device, compiles the standard
//      kernel's own source (embedded in the library at build time) with that
//      expression as its score_mod using NVRTC, for sm_103a, into a cubin;
//   3. loads the cubin into the current context and launches it exactly like
//      the built-in standard kernel (same parameters, same tensor maps).
// NVRTC is loaded on first use (dlopen), so the library has no link-time
// dependency on it; without it FL_MOD_EXPR returns FL_ERR_UNSUPPORTED.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <dlfcn.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <type_traits>
#include <vector>

#include "launch.h"
#include "jit_sources.inc" // kJitSources: {file name, text} of the kernel sources

namespace fl {
namespace {

void put(char *dst, size_t n, const char *fmt, ...)
{
    if (!dst || n == 0)
        return;
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(dst, n, fmt, ap);
    va_end(ap);
}

// ------------------------------------------------------------------ grammar
//
//   expr    := sum [ relop sum ]          relop: < <= > >= == !=  (no chaining)
//   sum     := term { (+|-) term }
//   term    := unary { (*|/) unary }
//   unary   := (-|+) unary | primary
//   primary := number | variable | inf | func ( expr {, expr} ) | ( expr )
//   variable: score b h q_idx kv_idx      func: see kFuncs
// A comparison yields 1 or 0.  Every value is fp32.

struct Func {
    const char *name;
    int arity;
};
constexpr Func kFuncs[] = {{"tanh", 1}, {"exp", 1},  {"exp2", 1}, {"log", 1},
                           {"log2", 1}, {"sqrt", 1}, {"abs", 1},  {"floor", 1},
                           {"min", 2},  {"max", 2},  {"where", 3}};
constexpr const char *kVars[] = {"score", "b", "h", "q_idx", "kv_idx"};
constexpr int kMaxDepth = 64;
constexpr size_t kMaxLen = 4096;

// A translated subexpression: its fp32 CUDA value and its derivative with
// respect to `score` (forward-mode differentiation carried through the
// parse), `zero` when the derivative is identically 0.
struct Dual {
    std::string v, d;
    bool zero = true;
};

Dual constant(const std::string &v)
{
    Dual r;
    r.v = v;
    r.d = "0.0f";
    return r;
}

class Translator {
  public:
    explicit Translator(const char *src) : s_(src) {}

    bool run(Dual &out, std::string &err)
    {
        if (strlen(s_) > kMaxLen) {
            err = "expression longer than 4096 characters";
            return false;
        }
        Dual o;
        if (expr(o)) {
            skip();
            if (s_[i_] == '\0') {
                out = o;
                return true;
            }
            fail("unexpected character");
        }
        err = err_;
        return false;
    }

  private:
    const char *s_;
    size_t i_ = 0;
    int depth_ = 0;
    std::string err_;

    void skip()
    {
        while (s_[i_] == ' ' || s_[i_] == '\t' || s_[i_] == '\n' || s_[i_] == '\r')
            ++i_;
    }
    bool fail(const char *what)
    {
        if (err_.empty()) {
            char buf[160];
            snprintf(buf, sizeof buf, "%s at offset %zu", what, i_);
            err_ = buf;
        }
        return false;
    }
    static bool is_alpha(char c) { return (c >= 'a' && c <= 'z') || (c >= 'A' && c <= 'Z') || c == '_'; }
    static bool is_digit(char c) { return c >= '0' && c <= '9'; }

    // which relational operator starts at i_ (0 if none)
    const char *relop() const
    {
        static const char *ops[] = {"<=", ">=", "==", "!=", "<", ">"};
        for (const char *op : ops)
            if (strncmp(s_ + i_, op, strlen(op)) == 0)
                return op;
        return nullptr;
    }

    bool expr(Dual &o)
    {
        if (++depth_ > kMaxDepth)
            return fail("expression nested too deeply");
        Dual a;
        if (!sum(a))
            return false;
        skip();
        if (const char *op = relop()) {
            i_ += strlen(op);
            Dual b;
            if (!sum(b))
                return false;
            skip();
            if (relop())
                return fail("comparisons do not chain (parenthesise one side)");
            o = constant("fl_x_bool(" + a.v + " " + op + " " + b.v + ")"); // piecewise constant
        } else {
            o = a;
        }
        --depth_;
        return true;
    }

    bool sum(Dual &o)
    {
        if (!term(o))
            return false;
        for (;;) {
            skip();
            const char c = s_[i_];
            if (c != '+' && c != '-')
                return true;
            ++i_;
            Dual b;
            if (!term(b))
                return false;
            Dual r;
            r.v = "(" + o.v + " " + c + " " + b.v + ")";
            r.zero = o.zero && b.zero;
            r.d = r.zero ? "0.0f" : "(" + o.d + " " + c + " " + b.d + ")";
            o = r;
        }
    }

    bool term(Dual &o)
    {
        if (!unary(o))
            return false;
        for (;;) {
            skip();
            const char c = s_[i_];
            if (c != '*' && c != '/')
                return true;
            if (s_[i_ + 1] == '*' || s_[i_ + 1] == '/')
                return fail("'**', '//' and comments are not part of the grammar");
            ++i_;
            Dual b;
            if (!unary(b))
                return false;
            Dual r;
            r.v = "(" + o.v + " " + c + " " + b.v + ")";
            r.zero = o.zero && b.zero;
            if (r.zero)
                r.d = "0.0f";
            else if (c == '*')
                r.d = "(" + o.d + " * " + b.v + " + " + o.v + " * " + b.d + ")";
            else
                r.d = "((" + o.d + " * " + b.v + " - " + o.v + " * " + b.d + ") / (" + b.v + " * " + b.v + "))";
            o = r;
        }
    }

    bool unary(Dual &o)
    {
        skip();
        const char c = s_[i_];
        if (c == '-' || c == '+') {
            ++i_;
            if (++depth_ > kMaxDepth)
                return fail("expression nested too deeply");
            Dual a;
            if (!unary(a))
                return false;
            --depth_;
            o.v = std::string("(") + c + a.v + ")";
            o.zero = a.zero;
            o.d = a.zero ? "0.0f" : std::string("(") + c + a.d + ")";
            return true;
        }
        return primary(o);
    }

    bool number(Dual &o)
    {
        const size_t start = i_;
        bool dot = false, exp = false;
        while (is_digit(s_[i_]))
            ++i_;
        if (s_[i_] == '.') {
            dot = true;
            ++i_;
            while (is_digit(s_[i_]))
                ++i_;
        }
        if (i_ == start + (dot ? 1 : 0))
            return fail("malformed number");
        if (s_[i_] == 'e' || s_[i_] == 'E') {
            exp = true;
            ++i_;
            if (s_[i_] == '+' || s_[i_] == '-')
                ++i_;
            if (!is_digit(s_[i_]))
                return fail("malformed exponent");
            while (is_digit(s_[i_]))
                ++i_;
        }
        if (is_alpha(s_[i_]) || s_[i_] == '.')
            return fail("malformed number");
        std::string t(s_ + start, i_ - start);
        if (!dot && !exp)
            t += ".0";
        else if (t.back() == '.')
            t += "0";
        o = constant("(" + t + "f)");
        return true;
    }

    // f(args) with its derivative: the chain rule through each function
    static Dual apply(const std::string &name, const std::vector<Dual> &a)
    {
        Dual r;
        std::string call = "fl_x_" + name + "(";
        for (size_t k = 0; k < a.size(); ++k)
            call += a[k].v + (k + 1 < a.size() ? ", " : ")");
        r.v = call;
        bool z = true;
        for (const Dual &x : a)
            z = z && x.zero;
        if (name == "floor")
            z = true;               // piecewise constant
        if (name == "where")
            z = a[1].zero && a[2].zero; // the condition is piecewise constant
        r.zero = z;
        if (z) {
            r.d = "0.0f";
            return r;
        }
        const std::string &u = a[0].v, &du = a[0].d;
        if (name == "tanh")
            r.d = "fl_dx_tanh(" + u + ", " + du + ")";
        else if (name == "exp")
            r.d = "(" + r.v + " * " + du + ")";
        else if (name == "exp2")
            r.d = "(" + r.v + " * 0.6931471805599453f * " + du + ")";
        else if (name == "log")
            r.d = "(" + du + " / " + u + ")";
        else if (name == "log2")
            r.d = "(" + du + " / (" + u + " * 0.6931471805599453f))";
        else if (name == "sqrt")
            r.d = "(" + du + " / (2.0f * " + r.v + "))";
        else if (name == "abs")
            r.d = "fl_x_where(fl_x_bool(" + u + " >= 0.0f), " + du + ", -" + du + ")";
        else if (name == "min")
            r.d = "fl_x_where(fl_x_bool(" + u + " <= " + a[1].v + "), " + du + ", " + a[1].d + ")";
        else if (name == "max")
            r.d = "fl_x_where(fl_x_bool(" + u + " >= " + a[1].v + "), " + du + ", " + a[1].d + ")";
        else // where(c, x, y)
            r.d = "fl_x_where(" + a[0].v + ", " + a[1].d + ", " + a[2].d + ")";
        return r;
    }

    bool primary(Dual &o)
    {
        skip();
        const char c = s_[i_];
        if (is_digit(c) || (c == '.' && is_digit(s_[i_ + 1])))
            return number(o);
        if (c == '(') {
            ++i_;
            Dual a;
            if (!expr(a))
                return false;
            skip();
            if (s_[i_] != ')')
                return fail("expected ')'");
            ++i_;
            o.v = "(" + a.v + ")";
            o.d = a.zero ? "0.0f" : "(" + a.d + ")";
            o.zero = a.zero;
            return true;
        }
        if (!is_alpha(c))
            return fail(c ? "unexpected character" : "unexpected end of expression");
        const size_t start = i_;
        while (is_alpha(s_[i_]) || is_digit(s_[i_]))
            ++i_;
        const std::string name(s_ + start, i_ - start);
        for (const char *v : kVars)
            if (name == v) {
                o = constant(name);
                if (name == "score") {
                    o.d = "1.0f";
                    o.zero = false;
                }
                return true;
            }
        if (name == "inf") {
            o = constant("fl_x_inf()");
            return true;
        }
        for (const Func &f : kFuncs) {
            if (name != f.name)
                continue;
            skip();
            if (s_[i_] != '(')
                return fail("expected '(' after a function name");
            ++i_;
            std::vector<Dual> args;
            for (int a = 0; a < f.arity; ++a) {
                Dual arg;
                if (!expr(arg))
                    return false;
                skip();
                if (s_[i_] != (a + 1 < f.arity ? ',' : ')'))
                    return fail(a + 1 < f.arity ? "expected ',' (too few arguments)"
                                                : "expected ')' (too many arguments)");
                ++i_;
                args.push_back(arg);
            }
            o = apply(name, args);
            return true;
        }
        i_ = start;
        return fail("unknown name");
    }
};

// ------------------------------------------------------------------ NVRTC

typedef int nvrtcResult_t;
typedef struct _nvrtcProgram *nvrtcProgram_t;
struct Nvrtc {
    nvrtcResult_t (*create)(nvrtcProgram_t *, const char *, const char *, int, const char *const *,
                            const char *const *);
    nvrtcResult_t (*destroy)(nvrtcProgram_t *);
    nvrtcResult_t (*compile)(nvrtcProgram_t, int, const char *const *);
    nvrtcResult_t (*log_size)(nvrtcProgram_t, size_t *);
    nvrtcResult_t (*log)(nvrtcProgram_t, char *);
    nvrtcResult_t (*cubin_size)(nvrtcProgram_t, size_t *);
    nvrtcResult_t (*cubin)(nvrtcProgram_t, char *);
    nvrtcResult_t (*add_name)(nvrtcProgram_t, const char *);
    nvrtcResult_t (*lowered)(nvrtcProgram_t, const char *, const char **);
    bool ok = false;
};

std::string cuda_home()
{
    for (const char *v : {"CUDA_HOME", "CUDA_PATH"})
        if (const char *e = getenv(v))
            if (*e)
                return e;
    return "/usr/local/cuda";
}

const Nvrtc &nvrtc()
{
    static Nvrtc n;
    static std::once_flag once;
    std::call_once(once, [] {
        const std::string home = cuda_home();
        const std::string cands[] = {"libnvrtc.so.13", home + "/lib64/libnvrtc.so.13",
                                     home + "/lib64/libnvrtc.so", "libnvrtc.so"};
        void *h = nullptr;
        for (const std::string &c : cands)
            if ((h = dlopen(c.c_str(), RTLD_NOW | RTLD_LOCAL)))
                break;
        if (!h)
            return;
        bool all = true;
        auto sym = [&](auto &fn, const char *name) {
            fn = reinterpret_cast<std::remove_reference_t<decltype(fn)>>(dlsym(h, name));
            all = all && fn;
        };
        sym(n.create, "nvrtcCreateProgram");
        sym(n.destroy, "nvrtcDestroyProgram");
        sym(n.compile, "nvrtcCompileProgram");
        sym(n.log_size, "nvrtcGetProgramLogSize");
        sym(n.log, "nvrtcGetProgramLog");
        sym(n.cubin_size, "nvrtcGetCUBINSize");
        sym(n.cubin, "nvrtcGetCUBIN");
        sym(n.add_name, "nvrtcAddNameExpression");
        sym(n.lowered, "nvrtcGetLoweredName");
        n.ok = all;
    });
    return n;
}

// The helpers every translated expression calls.
const char *kHelpers =
    "#define FL_SCORE_EXPR 1\n"
    "__device__ __forceinline__ float fl_x_bool(bool c) { return c ? 1.f : 0.f; }\n"
    "__device__ __forceinline__ float fl_x_inf() { return __int_as_float(0x7f800000); }\n"
    // exponentials on the hardware 2^x (relative error ~2^-22);
    // tanh(x) = 1 - 2 / (1 + e^(2x)) on it and the hardware
    // reciprocal (absolute error ~1e-7; +-1 at the extremes)
    "__device__ __forceinline__ float fl_x_exp2(float x)\n"
    "{ float y; asm(\"ex2.approx.ftz.f32 %0, %1;\" : \"=f\"(y) : \"f\"(x)); return y; }\n"
    "__device__ __forceinline__ float fl_x_exp(float x) { return fl_x_exp2(x * 1.4426950408889634f); }\n"
    "__device__ __forceinline__ float fl_x_tanh(float x)\n"
    "{\n"
    "    float r;\n"
    "    asm(\"rcp.approx.ftz.f32 %0, %1;\" : \"=f\"(r) : \"f\"(1.f + fl_x_exp2(x * 2.8853900817779268f)));\n"
    "    return 1.f - 2.f * r;\n"
    "}\n"
    "__device__ __forceinline__ float fl_x_log(float x) { return logf(x); }\n"
    "__device__ __forceinline__ float fl_x_log2(float x) { return log2f(x); }\n"
    "__device__ __forceinline__ float fl_x_sqrt(float x) { return sqrtf(x); }\n"
    "__device__ __forceinline__ float fl_x_abs(float x) { return fabsf(x); }\n"
    "__device__ __forceinline__ float fl_x_floor(float x) { return floorf(x); }\n"
    "__device__ __forceinline__ float fl_x_min(float x, float y) { return fminf(x, y); }\n"
    "__device__ __forceinline__ float fl_x_max(float x, float y) { return fmaxf(x, y); }\n"
    "__device__ __forceinline__ float fl_x_where(float c, float x, float y) { return c != 0.f ? x : y; }\n"
    "__device__ __forceinline__ float fl_dx_tanh(float x, float dx)\n"
    "{ const float t = fl_x_tanh(x); return (1.f - t * t) * dx; }\n";

std::string expr_function(const char *name, const std::string &body)
{
    return std::string("__device__ __forceinline__ float ") + name +
           "(float score, float b, float h, float q_idx, float kv_idx)\n"
           "{\n"
           "    (void)score; (void)b; (void)h; (void)q_idx; (void)kv_idx;\n"
           "    return " + body + ";\n"
           "}\n";
}

// The forward: the standard kernel's source with the expression as its
// score_mod.
std::string forward_source(const std::string &cuda)
{
    return std::string(kHelpers) + expr_function("fl_score_expr", cuda) + "#include \"fwd_standard.cu\"\n";
}

// The backward: the backward kernels' source with the expression and its
// derivative with respect to the score.
std::string backward_source(const std::string &cuda, const std::string &grad)
{
    return std::string(kHelpers) + expr_function("fl_score_expr", cuda) +
           expr_function("fl_score_expr_du", grad) + "#include \"bwd_standard.cu\"\n";
}

// MOD_EXPR at head dimension D
std::vector<std::string> forward_kernels(int D)
{
    return {"fl::std_fwd_kernel<3, " + std::to_string(D) + ">"};
}
const std::vector<std::string> kBackwardKernels = {"fl::bwd_fused_kernel<3>"}; // dK/dV and dQ tiles

// Compiles `src` (which includes the embedded kernel sources) for sm_103a;
// the cubin and the mangled names of `kernels` on success.
bool compile(const std::string &src, const std::vector<std::string> &kernels, std::vector<char> &cubin,
             std::vector<std::string> &names, char *err, size_t err_n)
{
    const Nvrtc &n = nvrtc();
    if (!n.ok) {
        put(err, err_n, "the runtime compiler (libnvrtc.so.13) was not found");
        return false;
    }
    std::vector<const char *> hnames, htexts;
    for (const auto &s : kJitSources) {
        hnames.push_back(s.name);
        htexts.push_back(s.text);
    }
    nvrtcProgram_t prog = nullptr;
    if (n.create(&prog, src.c_str(), "score_expr_kernel.cu", int(hnames.size()), htexts.data(),
                 hnames.data()) != 0) {
        put(err, err_n, "nvrtcCreateProgram failed");
        return false;
    }
    for (const std::string &k : kernels)
        n.add_name(prog, k.c_str());
    const std::string inc = "--include-path=" + cuda_home() + "/include";
    // --prec-div=false: '/' is the fast division (within 2 ulp), not the
    // IEEE-rounded one, whose slow path would cost ~10 instructions a score
    const char *opts[] = {"--gpu-architecture=sm_103a", "-std=c++17", "-lineinfo", "--prec-div=false",
                          inc.c_str()};
    const int rc = n.compile(prog, 5, opts);
    bool good = rc == 0;
    if (!good) {
        size_t ls = 0;
        n.log_size(prog, &ls);
        std::string log(ls, '\0');
        if (ls)
            n.log(prog, &log[0]);
        put(err, err_n, "runtime compilation failed: %.900s", log.c_str());
    } else {
        size_t cs = 0;
        good = n.cubin_size(prog, &cs) == 0 && cs > 0;
        names.clear();
        for (const std::string &k : kernels) {
            const char *lowered = nullptr;
            good = good && n.lowered(prog, k.c_str(), &lowered) == 0 && lowered;
            if (good)
                names.push_back(lowered);
        }
        if (good) {
            cubin.resize(cs);
            good = n.cubin(prog, cubin.data()) == 0;
        }
        if (!good)
            put(err, err_n, "reading the compiled kernel failed");
    }
    n.destroy(&prog);
    return good;
}

// ------------------------------------------------------------------ modules

struct Driver {
    PFN_cuModuleLoadData_v2000 load = nullptr;
    PFN_cuModuleGetFunction_v2000 get = nullptr;
    PFN_cuFuncGetAttribute_v2020 attr = nullptr;
    PFN_cuFuncSetAttribute_v9000 set = nullptr;
    PFN_cuLaunchKernel_v4000 launch = nullptr;
    bool ok = false;
};

const Driver &driver()
{
    static Driver d;
    static std::once_flag once;
    std::call_once(once, [] {
        auto entry = [](const char *name, int ver) -> void * {
            void *f = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion(name, &f, ver, cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess)
                return nullptr;
            return f;
        };
        d.load = reinterpret_cast<PFN_cuModuleLoadData_v2000>(entry("cuModuleLoadData", 2000));
        d.get = reinterpret_cast<PFN_cuModuleGetFunction_v2000>(entry("cuModuleGetFunction", 2000));
        d.attr = reinterpret_cast<PFN_cuFuncGetAttribute_v2020>(entry("cuFuncGetAttribute", 2020));
        d.set = reinterpret_cast<PFN_cuFuncSetAttribute_v9000>(entry("cuFuncSetAttribute", 9000));
        d.launch = reinterpret_cast<PFN_cuLaunchKernel_v4000>(entry("cuLaunchKernel", 4000));
        d.ok = d.load && d.get && d.attr && d.set && d.launch;
    });
    return d;
}

// One loaded kernel per (device, translated expression); modules stay loaded
// until the process exits.
std::mutex g_mutex;
std::map<std::pair<int, std::string>, CUfunction> g_kernels;

} // namespace

bool score_expr_translate(const char *expr, char *cuda, size_t n, char *err, size_t err_n)
{
    return score_expr_translate_grad(expr, cuda, n, nullptr, 0, err, err_n);
}

bool score_expr_translate_grad(const char *expr, char *cuda, size_t n, char *grad, size_t grad_n, char *err,
                               size_t err_n)
{
    if (!expr) {
        put(err, err_n, "no expression");
        return false;
    }
    Dual out;
    std::string e;
    if (!Translator(expr).run(out, e)) {
        put(err, err_n, "%s", e.c_str());
        return false;
    }
    if (out.v.size() + 1 > n || (grad && out.d.size() + 1 > grad_n)) {
        put(err, err_n, "translated expression too long");
        return false;
    }
    memcpy(cuda, out.v.c_str(), out.v.size() + 1);
    if (grad)
        memcpy(grad, out.d.c_str(), out.d.size() + 1);
    return true;
}

bool score_expr_compile_only(const char *cuda, const char *grad, char *err, size_t err_n)
{
    std::vector<char> cubin;
    std::vector<std::string> names;
    return compile(forward_source(cuda), forward_kernels(64), cubin, names, err, err_n) &&
           (!grad || compile(backward_source(cuda, grad), kBackwardKernels, cubin, names, err, err_n));
}

cudaError_t launch_standard_expr(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                                 const StdParams &p, int grid, cudaStream_t stream, const char *cuda,
                                 char *err, size_t err_n)
{
    const Driver &d = driver();
    if (!d.ok) {
        put(err, err_n, "driver entry points for module loading are unavailable");
        return cudaErrorNotSupported;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const size_t smem = standard_smem_bytes(p.head_dim);
    const std::string key = std::to_string(p.head_dim) + ":" + cuda;
    CUfunction fn = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        auto it = g_kernels.find({dev, key});
        if (it != g_kernels.end()) {
            fn = it->second;
        } else {
            std::vector<char> cubin;
            std::vector<std::string> names;
            if (!compile(forward_source(cuda), forward_kernels(p.head_dim), cubin, names, err, err_n))
                return cudaErrorInvalidSource;
            // the runtime has made the device's primary context current
            if ((e = cudaFree(nullptr)) != cudaSuccess)
                return e;
            CUmodule mod = nullptr;
            if (d.load(&mod, cubin.data()) != CUDA_SUCCESS || d.get(&fn, mod, names[0].c_str()) != CUDA_SUCCESS) {
                put(err, err_n, "loading the compiled kernel failed");
                return cudaErrorInvalidKernelImage;
            }
            // the setmaxnreg split assumes exactly kStdRegs registers at launch
            int regs = 0;
            if (d.attr(&regs, CU_FUNC_ATTRIBUTE_NUM_REGS, fn) != CUDA_SUCCESS || regs != kStdRegs) {
                put(err, err_n, "the compiled kernel uses %d registers per thread, not %d", regs, kStdRegs);
                return cudaErrorInvalidConfiguration;
            }
            if (d.set(fn, CU_FUNC_ATTRIBUTE_MAX_DYNAMIC_SHARED_SIZE_BYTES, int(smem)) != CUDA_SUCCESS) {
                put(err, err_n, "setting the kernel's shared-memory size failed");
                return cudaErrorInvalidConfiguration;
            }
            g_kernels[{dev, key}] = fn;
        }
    }
    void *args[] = {const_cast<CUtensorMap *>(&tq), const_cast<CUtensorMap *>(&tk),
                    const_cast<CUtensorMap *>(&tv), const_cast<StdParams *>(&p)};
    if (d.launch(fn, unsigned(grid), 1, 1, unsigned(kStdThreads), 1, 1, unsigned(smem),
                 reinterpret_cast<CUstream>(stream), args, nullptr) != CUDA_SUCCESS) {
        put(err, err_n, "launching the compiled kernel failed");
        return cudaErrorLaunchFailure;
    }
    return cudaSuccess;
}

// One loaded backward kernel per (device, expression).
std::map<std::pair<int, std::string>, CUfunction> g_bwd_kernels;

cudaError_t launch_bwd_expr(const CUtensorMap &tq, const CUtensorMap &tdo, const CUtensorMap &tk,
                            const CUtensorMap &tv, const CUtensorMap &tq128, const CUtensorMap &tdo128,
                            const CUtensorMap &tk128, const CUtensorMap &tv128, const BwdParams &p,
                            cudaStream_t stream, const char *cuda, const char *grad, char *err, size_t err_n)
{
    const Driver &d = driver();
    if (!d.ok) {
        put(err, err_n, "driver entry points for module loading are unavailable");
        return cudaErrorNotSupported;
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    const size_t smem = bwd_smem_bytes();
    CUfunction fn = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        const std::string key = std::string(cuda) + "\n" + grad;
        auto it = g_bwd_kernels.find({dev, key});
        if (it != g_bwd_kernels.end()) {
            fn = it->second;
        } else {
            std::vector<char> cubin;
            std::vector<std::string> names;
            if (!compile(backward_source(cuda, grad), kBackwardKernels, cubin, names, err, err_n))
                return cudaErrorInvalidSource;
            if ((e = cudaFree(nullptr)) != cudaSuccess)
                return e;
            CUmodule mod = nullptr;
            if (d.load(&mod, cubin.data()) != CUDA_SUCCESS || d.get(&fn, mod, names[0].c_str()) != CUDA_SUCCESS) {
                put(err, err_n, "loading the compiled backward kernel failed");
                return cudaErrorInvalidKernelImage;
            }
            if (d.set(fn, CU_FUNC_ATTRIBUTE_MAX_DYNAMIC_SHARED_SIZE_BYTES, int(smem)) != CUDA_SUCCESS) {
                put(err, err_n, "setting the backward kernel's shared-memory size failed");
                return cudaErrorInvalidConfiguration;
            }
            g_bwd_kernels[{dev, key}] = fn;
        }
    }
    // the parameter order of bwd_fused_kernel
    void *args[] = {const_cast<CUtensorMap *>(&tk128), const_cast<CUtensorMap *>(&tv128),
                    const_cast<CUtensorMap *>(&tq), const_cast<CUtensorMap *>(&tdo),
                    const_cast<CUtensorMap *>(&tq128), const_cast<CUtensorMap *>(&tdo128),
                    const_cast<CUtensorMap *>(&tk), const_cast<CUtensorMap *>(&tv), const_cast<BwdParams *>(&p)};
    const int64_t blocks = bwd_fused_blocks(p);
    if (d.launch(fn, unsigned(blocks), 1, 1, unsigned(kBwdThreads), 1, 1, unsigned(smem),
                 reinterpret_cast<CUstream>(stream), args, nullptr) != CUDA_SUCCESS) {
        put(err, err_n, "launching the compiled backward kernel failed");
        return cudaErrorLaunchFailure;
    }
    return cudaSuccess;
}

} // namespace fl
