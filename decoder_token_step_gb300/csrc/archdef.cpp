// archdef.cpp -- parser and validator of the .archdef text format.
//
// Format ("Local inference and architectures", synsema.dev, sections "The format", "Rules" and
// "The operations"): an `arch NAME` line that must equal the file name, `kind decoder`, optional
// `param KEY VALUE` lines, then three sections in order -- prologue, block (run once per layer with
// {i} replaced by the layer index), epilogue -- whose lines are `dst = op(args)` (assign to a
// register) or `op(dst, args)` (modify one in place). `#` starts a comment; blank lines are free.
//
// The vocabulary is closed: sixteen ops and nothing else. There is no control flow and no I/O, so
// any other word -- if, while, loop, for, exec, import, open, http, env, ... -- is an unknown op
// (section "No control flow, and that is the security property"). Errors name the file and line
// and suggest the nearest op (section "Errors"); a broken text is refused, never replaced by a
// built-in definition.
#include <algorithm>
#include <cctype>
#include <cstdlib>
#include <map>
#include <set>
#include <vector>
#include <sstream>

#include "syn_internal.h"

namespace syn {

const char *const kOps[16] = {"embed", "rms_norm", "matmul", "add_bias", "norm_heads", "rope",
                              "attention", "silu", "gelu", "gelu_tanh", "relu", "mul",
                              "add", "scale", "copy", "last"};

namespace {

// Argument kinds of each op's signature (after the destination in the in-place form).
// R = register, T = tensor name (may be "a | b"), C = head-count metadata name, S = scalar.
struct Sig { const char *op; const char *args; bool assign_only; bool inplace_ok; };
const Sig kSigs[] = {
    {"embed", "T", true, false},       {"rms_norm", "RT", false, true}, {"matmul", "RT", true, false},
    {"add_bias", "RT", false, true},   {"norm_heads", "RTC", false, true}, {"rope", "RC", false, true},
    {"attention", "RRR", true, false}, {"silu", "R", false, true},    {"gelu", "R", false, true},
    {"gelu_tanh", "R", false, true},   {"relu", "R", false, true},    {"mul", "RR", false, true},
    {"add", "RR", false, true},        {"scale", "RS", false, true},  {"copy", "R", true, false},
    {"last", "R", false, true},
};

const Sig *find_sig(const std::string &op) {
    for (const Sig &s : kSigs)
        if (op == s.op) return &s;
    return nullptr;
}

std::string trim(const std::string &s) {
    size_t a = 0, b = s.size();
    while (a < b && std::isspace((unsigned char)s[a])) ++a;
    while (b > a && std::isspace((unsigned char)s[b - 1])) --b;
    return s.substr(a, b - a);
}

int edit_distance(const std::string &a, const std::string &b) {
    std::vector<int> prev(b.size() + 1), cur(b.size() + 1);
    for (size_t j = 0; j <= b.size(); ++j) prev[j] = (int)j;
    for (size_t i = 1; i <= a.size(); ++i) {
        cur[0] = (int)i;
        for (size_t j = 1; j <= b.size(); ++j)
            cur[j] = std::min({prev[j] + 1, cur[j - 1] + 1, prev[j - 1] + (a[i - 1] != b[j - 1])});
        std::swap(prev, cur);
    }
    return prev[b.size()];
}

bool is_ident(const std::string &s) {
    if (s.empty() || !(std::isalpha((unsigned char)s[0]) || s[0] == '_')) return false;
    for (char c : s)
        if (!(std::isalnum((unsigned char)c) || c == '_')) return false;
    return true;
}

bool is_tensor_ref(const std::string &s) {
    // one or more GGUF names separated by '|': letters, digits, '_', '.', and the {i} placeholder
    std::stringstream ss(s);
    std::string part;
    int n = 0;
    while (std::getline(ss, part, '|')) {
        part = trim(part);
        if (part.empty()) return false;
        for (size_t i = 0; i < part.size(); ++i) {
            char c = part[i];
            if (c == '{') {
                if (part.compare(i, 3, "{i}") != 0) return false;
                i += 2;
                continue;
            }
            if (!(std::isalnum((unsigned char)c) || c == '_' || c == '.')) return false;
        }
        ++n;
    }
    return n > 0;
}

// " — did you mean `c`?" for the candidate nearest to w (edit distance at most 2 and shorter than
// w itself), else ""
std::string hint(const std::string &w, const std::vector<std::string> &cands) {
    std::string best;
    int bd = 1 << 30;
    for (const std::string &c : cands) {
        const int d = edit_distance(w, c);
        if (d < bd) {
            bd = d;
            best = c;
        }
    }
    if (best.empty() || bd > 2 || bd >= (int)w.size()) return "";
    return " \xe2\x80\x94 did you mean `" + best + "`?";
}

bool is_number(const std::string &s) {
    if (s.empty()) return false;
    char *end = nullptr;
    std::strtod(s.c_str(), &end);
    return end && *end == 0;
}

}  // namespace

bool parse_archdef(const std::string &file_arch, const std::string &text, Archdef &out, std::string &err) {
    const std::string file = (file_arch.empty() ? std::string("<archdef>") : file_arch) + ".archdef";
    auto fail = [&](int line, const std::string &msg) {
        err = file + ": line " + std::to_string(line) + ": " + msg;
        return false;
    };
    out = Archdef();
    int section = -1, line_no = 0, arch_line = 0;
    bool have_kind = false;
    std::set<std::string> defined;  // registers assigned so far (for use-before-definition)
    std::stringstream in(text);
    std::string raw;
    while (std::getline(in, raw)) {
        ++line_no;
        size_t hash = raw.find('#');
        std::string s = trim(hash == std::string::npos ? raw : raw.substr(0, hash));
        if (s.empty()) continue;
        std::stringstream ws(s);
        std::string w0;
        ws >> w0;
        if (w0 == "arch") {
            std::string name, extra;
            ws >> name >> extra;
            if (name.empty() || !extra.empty() || !is_ident(name)) return fail(line_no, "expected `arch NAME`");
            if (!out.arch.empty()) return fail(line_no, "second `arch` line");
            if (section >= 0) return fail(line_no, "`arch` must come before the sections");
            out.arch = name;
            arch_line = line_no;
            continue;
        }
        if (w0 == "kind") {
            std::string k, extra;
            ws >> k >> extra;
            if (k != "decoder" || !extra.empty()) return fail(line_no, "only `kind decoder` is supported" + hint(k, {"decoder"}));
            have_kind = true;
            continue;
        }
        if (w0 == "param") {
            std::string key, val, extra;
            ws >> key >> val >> extra;
            if (key.empty() || val.empty() || !extra.empty()) return fail(line_no, "expected `param KEY VALUE`");
            if (section >= 0) return fail(line_no, "`param` must come before the sections");
            if (key == "window_pattern") {
                if (!is_number(val) || std::atoi(val.c_str()) < 1) return fail(line_no, "window_pattern must be a positive integer");
                out.window_pattern = std::atoi(val.c_str());
            } else if (key == "rope_pairs") {
                if (val != "adjacent" && val != "half")
                    return fail(line_no, "rope_pairs must be `adjacent` or `half`" + hint(val, {"adjacent", "half"}));
                out.rope_adjacent = val == "adjacent";
            } else {
                return fail(line_no, "unknown param `" + key + "` (known: window_pattern, rope_pairs)" +
                                         hint(key, {"window_pattern", "rope_pairs"}));
            }
            continue;
        }
        if (s == "prologue" || s == "block" || s == "epilogue") {
            int want = s == "prologue" ? 0 : s == "block" ? 1 : 2;
            if (want <= section) return fail(line_no, "section `" + s + "` out of order (prologue, block, epilogue)");
            section = want;
            continue;
        }
        // a statement: [dst =] op(args)
        Step st;
        st.line = line_no;
        std::string call = s;
        size_t eq = s.find('=');
        size_t lp0 = s.find('(');
        if (eq != std::string::npos && (lp0 == std::string::npos || eq < lp0)) {
            st.dst = trim(s.substr(0, eq));
            st.assign = true;
            call = trim(s.substr(eq + 1));
            if (!is_ident(st.dst)) return fail(line_no, "bad register name `" + st.dst + "`");
        }
        size_t lp = call.find('('), rp = call.rfind(')');
        std::string opname = trim(lp == std::string::npos ? call : call.substr(0, lp));
        // the op name first: an unknown word is the error to report, whatever follows it
        const Sig *sig = find_sig(opname);
        if (!sig) {
            // a bare word is more likely a misspelt section header than an operation
            const bool bare = !st.assign && lp == std::string::npos;
            std::vector<std::string> cands;
            if (bare) cands = {"prologue", "block", "epilogue"};
            std::string h = hint(opname, cands);
            if (h.empty()) {
                cands.clear();
                for (const char *o : kOps) cands.push_back(o);
                h = hint(opname, cands);
            }
            return fail(line_no, (bare ? "unknown section or operation `" : "unknown operation `") + opname + "`" + h);
        }
        if (section < 0) return fail(line_no, "statement before any section");
        if (lp == std::string::npos || rp == std::string::npos || rp < lp || trim(call.substr(rp + 1)) != "")
            return fail(line_no, "expected `" + opname + "(...)`");
        st.op = opname;
        std::string inner = call.substr(lp + 1, rp - lp - 1);
        if (!trim(inner).empty()) {
            std::stringstream as(inner);
            std::string a;
            while (std::getline(as, a, ',')) st.args.push_back(trim(a));
        }
        if (!st.assign) {
            if (!sig->inplace_ok) return fail(line_no, "`" + opname + "` needs a destination: `dst = " + opname + "(...)`");
            if (st.args.empty()) return fail(line_no, "`" + opname + "` needs a register to modify");
            st.dst = st.args[0];
        }
        const std::string kinds = sig->args;
        if (st.args.size() != kinds.size())
            return fail(line_no, "`" + opname + "` takes " + std::to_string(kinds.size()) + " argument(s), got " +
                                     std::to_string(st.args.size()));
        for (size_t i = 0; i < kinds.size(); ++i) {
            const std::string &a = st.args[i];
            bool ok = kinds[i] == 'R' ? is_ident(a) : kinds[i] == 'T' ? is_tensor_ref(a)
                    : kinds[i] == 'C' ? is_ident(a) : (is_number(a) || is_ident(a));
            if (!ok) return fail(line_no, "argument " + std::to_string(i + 1) + " of `" + opname + "` is malformed: `" + a + "`");
            if (kinds[i] == 'R' && !defined.count(a))
                return fail(line_no, "register `" + a + "` is read before it is assigned" +
                                         hint(a, std::vector<std::string>(defined.begin(), defined.end())));
        }
        if (opname == "attention" && section != 1) return fail(line_no, "`attention` is only allowed in the block");
        if (st.assign) defined.insert(st.dst);
        out.sec[section].push_back(st);
    }
    if (out.arch.empty()) return fail(line_no ? line_no : 1, "missing `arch NAME` line");
    if (!have_kind) return fail(arch_line, "missing `kind decoder` line");
    if (!file_arch.empty() && out.arch != file_arch)
        return fail(arch_line, "declares `arch " + out.arch + "`; the file name says `" + file_arch + "`");
    if (out.sec[1].empty()) return fail(line_no, "empty or missing `block` section");
    if (!defined.count("logits")) return fail(line_no, "no step assigns register `logits`");
    if (!defined.count("x")) return fail(line_no, "no step assigns register `x` (the residual)");
    return true;
}

}  // namespace syn
