// Host pack planner and result collection.
//
// The layout follows "spinf-serve 0.1.1" (PyPI project page), "What it does"
// and "Speed and scale": each content is read once, each question is a branch of
// the same pass that sees its own content and its own tokens, never a sibling or
// another packed input; inputs are packed into passes of --token-budget rows
// ("spinf-serve" man page, PARAMETERS); long inputs run alone, split with the
// content repeated (man page, CAVEATS).  Options form a token trie per question
// (PyPI page, "Layout": "templates to token tries").  A searched slot ({*}, {n},
// {$}; PyPI page, "What it does") lays out its template only and is scored at its
// last template row.  A placeholder grid (same section: placeholders turn one
// template into a grid of questions) is expanded into one question per
// combination of placeholder values before anything else.
//
// Visibility is encoded by two integers per row: key k is visible to exactly the
// rows [k, end[k]) -- in a pre-order layout a row's descendants follow it
// contiguously -- and pos[] is the depth on the root path.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <deque>
#include <memory>
#include <new>
#include <string>
#include <unordered_map>
#include <vector>

#include "internal.h"

namespace spinf {

thread_local std::string g_last_error;

spinf_status fail(spinf_status s, const std::string& msg) {
    g_last_error = msg;
    return s;
}
spinf_status ok() { return SPINF_OK; }

namespace {

// One question's option trie: nodes are proper prefixes of options.
struct Trie {
    std::vector<int32_t> tok;                   // token of each node
    std::vector<int32_t> depth;                 // 1 for a child of the slot
    std::vector<std::vector<int32_t>> kids;     // children in insertion order
    std::vector<int32_t> root_kids;
    std::vector<int32_t> order;                 // nodes in pre-order
    std::vector<int32_t> rank;                  // node -> index in pre-order
    std::vector<int32_t> subtree;               // node -> nodes in its subtree (itself included)
    std::vector<std::vector<int32_t>> opt_node; // option, token i >= 1 -> node of prefix [0, i)
};

void build_trie(const spinf_question& q, Trie& t) {
    bool single = true;   // single-token options only: no node, and the layout reads no opt_node
    for (int32_t o = 0; o < q.n_options && single; ++o) single = q.options[o].n == 1;
    if (single) return;
    t.opt_node.resize(q.n_options);
    for (int32_t o = 0; o < q.n_options; ++o) {
        const spinf_tokens& opt = q.options[o];
        t.opt_node[o].assign(opt.n, -1);
        int32_t cur = -1;
        for (int32_t i = 0; i + 1 < opt.n; ++i) {
            std::vector<int32_t>& kids = cur < 0 ? t.root_kids : t.kids[cur];
            int32_t found = -1;
            for (int32_t c : kids)
                if (t.tok[c] == opt.ids[i]) { found = c; break; }
            if (found < 0) {
                found = (int32_t)t.tok.size();
                t.tok.push_back(opt.ids[i]);
                t.depth.push_back(cur < 0 ? 1 : t.depth[cur] + 1);
                t.kids.emplace_back();
                (cur < 0 ? t.root_kids : t.kids[cur]).push_back(found);
            }
            cur = found;
            t.opt_node[o][i + 1] = cur;
        }
    }
    // pre-order with an explicit stack
    std::vector<int32_t> stack(t.root_kids.rbegin(), t.root_kids.rend());
    while (!stack.empty()) {
        int32_t n = stack.back();
        stack.pop_back();
        t.order.push_back(n);
        for (auto it = t.kids[n].rbegin(); it != t.kids[n].rend(); ++it) stack.push_back(*it);
    }
    t.rank.assign(t.tok.size(), 0);
    for (size_t i = 0; i < t.order.size(); ++i) t.rank[t.order[i]] = (int32_t)i;
    t.subtree.assign(t.tok.size(), 1);
    for (size_t i = t.order.size(); i-- > 0;) {
        int32_t n = t.order[i];
        for (int32_t c : t.kids[n]) t.subtree[n] += t.subtree[c];
    }
}

// A floor is shared by the questions with the same template and the same option lists
// (in the same order): a 64-bit FNV-1a hash of those ids and lengths finds the
// candidates, and same_question decides.
uint64_t question_hash(const spinf_question& q) {
    uint64_t h = 14695981039346656037ull;
    auto put = [&](int32_t v) { h = (h ^ static_cast<uint32_t>(v)) * 1099511628211ull; };
    put(q.tmpl.n);
    for (int32_t i = 0; i < q.tmpl.n; ++i) put(q.tmpl.ids[i]);
    put(q.n_options);
    for (int32_t o = 0; o < q.n_options; ++o) {
        put(q.options[o].n);
        for (int32_t i = 0; i < q.options[o].n; ++i) put(q.options[o].ids[i]);
    }
    return h;
}

bool same_question(const spinf_question& a, const spinf_question& b) {
    if (a.tmpl.n != b.tmpl.n || a.n_options != b.n_options) return false;
    if (std::memcmp(a.tmpl.ids, b.tmpl.ids, sizeof(int32_t) * a.tmpl.n) != 0) return false;
    for (int32_t o = 0; o < a.n_options; ++o) {
        const spinf_tokens &x = a.options[o], &y = b.options[o];
        if (x.n != y.n || std::memcmp(x.ids, y.ids, sizeof(int32_t) * x.n) != 0) return false;
    }
    return true;
}

struct Unit {
    int32_t source;                       // user input, or -1 for a floor
    int32_t floor_id;                     // floor index, or -1
    spinf_tokens content;
    std::vector<const spinf_question*> qs;
    std::vector<const Trie*> tries;
    std::vector<int32_t> qidx;            // flat user-question index (floors: floor index)
    int64_t size;
};

// Grid cells as ordinary questions, appended after each input's own questions
// (first placeholder slowest).  The expanded inputs point into `store`.
struct Expanded {
    std::vector<spinf_input> inputs;
    std::vector<std::vector<spinf_question>> questions;
    std::deque<std::vector<int32_t>> templates;
};

spinf_status expand_grids(const spinf_input* inputs, int32_t n_inputs, const spinf_plan_opts& o, Expanded& x) {
    x.inputs.assign(inputs, inputs + n_inputs);
    x.questions.resize(n_inputs);
    for (int32_t i = 0; i < n_inputs; ++i) {
        const spinf_input& in = inputs[i];
        auto where = [i]() { return "input " + std::to_string(i); };   // built only for an error
        if (in.n_grids < 0 || (in.n_grids > 0 && !in.grids)) return fail(SPINF_E_INVALID, where() + ": bad grid array");
        if (in.n_questions < 0 || (in.n_questions > 0 && !in.questions))
            return fail(SPINF_E_INVALID, where() + ": bad arrays");
        int64_t total = in.n_questions;
        for (int32_t gi = 0; gi < in.n_grids; ++gi) {
            const spinf_grid& g = in.grids[gi];
            if (g.n_placeholders < 0 || !g.segments || (g.n_placeholders > 0 && (!g.values || !g.n_values)))
                return fail(SPINF_E_INVALID, where() + ": bad grid");
            int64_t cells = 1;
            for (int32_t p = 0; p < g.n_placeholders; ++p) {
                if (g.n_values[p] < 1) return fail(SPINF_E_INVALID, where() + ": a grid placeholder without values");
                cells = std::min<int64_t>(cells * g.n_values[p], (int64_t)1 << 40);
            }
            total += cells;
            if (total > o.max_prompts_per_input)
                return fail(SPINF_E_LIMIT, where() + ": more questions than max_prompts_per_input");
        }
        if (in.n_grids == 0) continue;
        std::vector<spinf_question>& qs = x.questions[i];
        qs.assign(in.questions, in.questions + in.n_questions);
        for (int32_t gi = 0; gi < in.n_grids; ++gi) {
            const spinf_grid& g = in.grids[gi];
            std::vector<int32_t> first(g.n_placeholders + 1, 0);   // first value of each placeholder
            for (int32_t p = 0; p < g.n_placeholders; ++p) first[p + 1] = first[p] + g.n_values[p];
            std::vector<int32_t> pick(g.n_placeholders, 0);          // odometer, last placeholder fastest
            for (;;) {
                std::vector<int32_t> t;
                auto put = [&](const spinf_tokens& s) {
                    if (s.n > 0 && s.ids) t.insert(t.end(), s.ids, s.ids + s.n);
                };
                put(g.segments[0]);
                for (int32_t p = 0; p < g.n_placeholders; ++p) {
                    put(g.values[first[p] + pick[p]]);
                    put(g.segments[p + 1]);
                }
                x.templates.push_back(std::move(t));
                spinf_question q{};
                q.tmpl.ids = x.templates.back().data();
                q.tmpl.n = (int32_t)x.templates.back().size();
                q.options = g.options;
                q.n_options = g.n_options;
                q.kind = g.kind;
                q.token_set = g.token_set;
                qs.push_back(q);
                int32_t p = g.n_placeholders - 1;
                while (p >= 0 && ++pick[p] == g.n_values[p]) pick[p--] = 0;
                if (p < 0) break;
            }
        }
        x.inputs[i].questions = qs.data();
        x.inputs[i].n_questions = (int32_t)qs.size();
        x.inputs[i].grids = nullptr;
        x.inputs[i].n_grids = 0;
    }
    return SPINF_OK;
}

bool ids_in_range(const spinf_tokens& t, int32_t vocab) {
    if (t.n > 0 && t.ids == nullptr) return false;
    if (vocab <= 0) return true;
    for (int32_t i = 0; i < t.n; ++i)
        if (t.ids[i] < 0 || t.ids[i] >= vocab) return false;
    return true;
}

}  // namespace

}  // namespace spinf

namespace spinf {

WindowSchedule& window_schedule(Pass& P, int32_t window) { return tile_schedule(P, window, kTile, kTile); }

// The schedule for window W (0: none) in KV tiles of `key_tile` keys (128, or 64: each
// input-anchored 128-key tile taken as its two halves) and Q tiles of `q_rows` rows (128, or 64:
// the halves of the planner's Q tiles): a KV tile stays iff some row of the Q tile sees one of
// its keys (within the window), in the planner's order.  Skipping a tile that no row sees
// changes no bit of the result.
WindowSchedule& tile_schedule(Pass& P, int32_t window, int32_t key_tile, int32_t q_rows) {
    for (auto& w : P.windows)
        if (w->window == window && w->key_tile == key_tile && w->q_rows == q_rows) return *w;
    auto ws = std::make_unique<WindowSchedule>();
    ws->window = window;
    ws->key_tile = key_tile;
    ws->q_rows = q_rows;
    const int32_t n_qt = P.T_pad / q_rows;
    ws->tile_ptr.assign(1, 0);
    int32_t mins[8][kTile];   // sparse table of pos over one Q tile's real rows
    for (int32_t qt = 0; qt < n_qt; ++qt) {
        const int32_t r0 = qt * q_rows, r1 = std::min(r0 + q_rows, P.T), nr = std::max(r1 - r0, 0);
        const int32_t qp = r0 / kTile;   // the planner's Q tile that holds these rows
        if (window > 0) {   // only the window test reads the table
            for (int32_t i = 0; i < nr; ++i) mins[0][i] = P.pos[r0 + i];
            for (int32_t l = 1; (1 << l) <= nr; ++l)
                for (int32_t i = 0; i + (1 << l) <= nr; ++i)
                    mins[l][i] = std::min(mins[l - 1][i], mins[l - 1][i + (1 << (l - 1))]);
        }
        auto range_min = [&](int32_t lo, int32_t hi) {   // rows [lo, hi) of the tile, hi > lo
            int32_t l = 0;
            while ((2 << l) <= hi - lo) ++l;
            return std::min(mins[l][lo - r0], mins[l][hi - r0 - (1 << l)]);
        };
        for (int32_t e = P.tile_ptr[qp]; e < P.tile_ptr[qp + 1]; ++e) {
            for (int32_t sub = 0; sub < kTile; sub += key_tile) {
                const int32_t kv0 = P.tile_kv[e] + sub, len = std::min(P.tile_len[e] - sub, key_tile);
                if (len <= 0) break;
                bool keep = false;
                for (int32_t k = kv0; k < kv0 + len && !keep; ++k) {   // rows that see k: [max(k, r0), min(end[k], r1))
                    const int32_t lo = std::max(k, r0), hi = std::min(P.end[k], r1);
                    keep = lo < hi && (window <= 0 || range_min(lo, hi) - P.pos[k] < window);
                }
                if (keep) {
                    ws->tile_kv.push_back(kv0);
                    ws->tile_len.push_back(len);
                }
            }
        }
        // a 64-row Q tile of pad rows only (the upper half of the last planner tile) keeps one
        // tile, masked for all its rows, so that the kernel writes its pad rows (as zeros)
        if (nr == 0 && ws->tile_kv.size() == (size_t)ws->tile_ptr.back() && P.tile_ptr[qp] < P.tile_ptr[qp + 1]) {
            ws->tile_kv.push_back(P.tile_kv[P.tile_ptr[qp]]);
            ws->tile_len.push_back(std::min(P.tile_len[P.tile_ptr[qp]], key_tile));
        }
        ws->tile_ptr.push_back((int32_t)ws->tile_kv.size());
    }
    std::vector<int32_t> order(n_qt);
    for (int32_t qt = 0; qt < n_qt; ++qt) order[qt] = qt;
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
        return ws->tile_ptr[a + 1] - ws->tile_ptr[a] > ws->tile_ptr[b + 1] - ws->tile_ptr[b];
    });
    ws->qt_work.assign(4 * (size_t)n_qt, 0);
    for (int32_t i = 0; i < n_qt; ++i) {
        ws->qt_work[4 * i] = order[i];
        ws->qt_work[4 * i + 1] = ws->tile_ptr[order[i]];
        ws->qt_work[4 * i + 2] = ws->tile_ptr[order[i] + 1] - ws->tile_ptr[order[i]];
    }
    P.windows.push_back(std::move(ws));
    return *P.windows.back();
}

}  // namespace spinf

using namespace spinf;

extern "C" void spinf_plan_opts_default(spinf_plan_opts* o) {
    if (!o) return;
    o->token_budget = 16384;
    o->max_tokens = 2000000;
    o->max_content_tokens = 4096;
    o->max_query_tokens = 256;
    o->max_options = 1000;
    o->max_option_tokens = 5;
    o->max_prompts_per_input = 10000;
    o->floors = 1;
    o->floor_prefix.ids = nullptr;
    o->floor_prefix.n = 0;
    o->vocab = 0;
    o->extract_k = 8;
}

extern "C" spinf_status spinf_pack_plan(const spinf_input* inputs, int32_t n_inputs,
                                        const spinf_plan_opts* opts_in, spinf_plan** out) {
    if (!out) return fail(SPINF_E_INVALID, "out is NULL");
    *out = nullptr;
    if (n_inputs < 0 || (n_inputs > 0 && !inputs)) return fail(SPINF_E_INVALID, "bad input array");
    spinf_plan_opts o;
    spinf_plan_opts_default(&o);
    if (opts_in) o = *opts_in;
    if (o.token_budget <= 0 || o.max_tokens <= 0 || o.floor_prefix.n < 0)
        return fail(SPINF_E_INVALID, "bad planner options");
    if (!ids_in_range(o.floor_prefix, o.vocab)) return fail(SPINF_E_INVALID, "floor prefix token out of range");
    if (o.extract_k < 1 || o.extract_k > 16) return fail(SPINF_E_INVALID, "extract_k must be in 1..16");

    try {
        // ---- grid cells become trailing questions of their input
        Expanded expanded;
        {
            spinf_status gs = expand_grids(inputs, n_inputs, o, expanded);
            if (gs) return gs;
            inputs = expanded.inputs.data();
        }

        // ---- validation and tries
        std::vector<std::vector<Trie>> tries(n_inputs);
        std::vector<std::vector<int64_t>> qsize(n_inputs);
        for (int32_t i = 0; i < n_inputs; ++i) {
            const spinf_input& in = inputs[i];
            auto where = [i]() { return "input " + std::to_string(i); };   // built only for an error
            if (in.content.n < 0 || in.n_questions < 0 || (in.n_questions > 0 && !in.questions))
                return fail(SPINF_E_INVALID, where() + ": bad arrays");
            if (in.content.n > o.max_content_tokens)
                return fail(SPINF_E_LIMIT, where() + ": content longer than max_content_tokens");
            if (in.n_questions > o.max_prompts_per_input)
                return fail(SPINF_E_LIMIT, where() + ": more questions than max_prompts_per_input");
            if (!ids_in_range(in.content, o.vocab)) return fail(SPINF_E_INVALID, where() + ": content token out of range");
            if (in.content.n == 0 && in.n_questions == 0) return fail(SPINF_E_INVALID, where() + ": nothing to read");
            int64_t size = in.content.n;
            tries[i].resize(in.n_questions);
            for (int32_t j = 0; j < in.n_questions; ++j) {
                const spinf_question& q = in.questions[j];
                auto wq = [&where, j]() { return where() + " question " + std::to_string(j); };
                if (q.tmpl.n <= 0) return fail(SPINF_E_INVALID, wq() + ": empty template");
                if (q.tmpl.n > o.max_query_tokens) return fail(SPINF_E_LIMIT, wq() + ": template longer than max_query_tokens");
                if (q.kind != SPINF_Q_SCORED && q.kind != SPINF_Q_SEARCHED) return fail(SPINF_E_INVALID, wq() + ": unknown kind");
                if (q.kind == SPINF_Q_SEARCHED) {   // template only: no options, no trie
                    if (q.n_options != 0) return fail(SPINF_E_INVALID, wq() + ": a searched slot has no options");
                    if (q.token_set < -1) return fail(SPINF_E_INVALID, wq() + ": bad token set");
                    if (!ids_in_range(q.tmpl, o.vocab)) return fail(SPINF_E_INVALID, wq() + ": template token out of range");
                    qsize[i].push_back(q.tmpl.n);
                    size += q.tmpl.n;
                    continue;
                }
                if (q.n_options <= 0 || !q.options) return fail(SPINF_E_INVALID, wq() + ": no options");
                if (q.n_options > o.max_options) return fail(SPINF_E_LIMIT, wq() + ": more options than max_options");
                for (int32_t a = 0; a < q.n_options; ++a) {
                    const spinf_tokens& opt = q.options[a];
                    if (opt.n <= 0 || !opt.ids) return fail(SPINF_E_INVALID, wq() + ": empty option");
                    if (opt.n > o.max_option_tokens) return fail(SPINF_E_LIMIT, wq() + ": option longer than max_option_tokens");
                    for (int32_t b = 0; b < a; ++b) {
                        const spinf_tokens& ob = q.options[b];
                        if (ob.n == opt.n && std::memcmp(ob.ids, opt.ids, sizeof(int32_t) * opt.n) == 0)
                            return fail(SPINF_E_INVALID, wq() + ": duplicate option");
                    }
                    if (!ids_in_range(opt, o.vocab)) return fail(SPINF_E_INVALID, wq() + ": option token out of range");
                }
                if (!ids_in_range(q.tmpl, o.vocab)) return fail(SPINF_E_INVALID, wq() + ": template token out of range");
                build_trie(q, tries[i][j]);
                qsize[i].push_back((int64_t)q.tmpl.n + (int64_t)tries[i][j].tok.size());
                size += qsize[i].back();
            }
            if (size > o.max_tokens) return fail(SPINF_E_LIMIT, where() + ": larger than max_tokens");
        }

        std::unique_ptr<spinf_plan> plan(new spinf_plan());

        // ---- units: user inputs (split when over budget), then floors
        std::vector<Unit> units;
        std::vector<int32_t> q_base(n_inputs + 1, 0);
        for (int32_t i = 0; i < n_inputs; ++i) q_base[i + 1] = q_base[i] + inputs[i].n_questions;
        for (int32_t i = 0; i < n_inputs; ++i) {
            const spinf_input& in = inputs[i];
            int64_t total = in.content.n;
            for (int64_t s : qsize[i]) total += s;
            if (total <= o.token_budget) {
                Unit u{i, -1, in.content, {}, {}, {}, total};
                for (int32_t j = 0; j < in.n_questions; ++j) {
                    u.qs.push_back(&in.questions[j]);
                    u.tries.push_back(&tries[i][j]);
                    u.qidx.push_back(q_base[i] + j);
                }
                units.push_back(std::move(u));
                continue;
            }
            if (in.n_questions == 0)
                return fail(SPINF_E_LIMIT, "input " + std::to_string(i) + ": content does not fit the token budget");
            int32_t j = 0;
            while (j < in.n_questions) {
                Unit u{i, -1, in.content, {}, {}, {}, in.content.n};
                while (j < in.n_questions && u.size + qsize[i][j] <= o.token_budget) {
                    u.size += qsize[i][j];
                    u.qs.push_back(&in.questions[j]);
                    u.tries.push_back(&tries[i][j]);
                    u.qidx.push_back(q_base[i] + j);
                    ++j;
                }
                if (u.qs.empty())
                    return fail(SPINF_E_LIMIT, "input " + std::to_string(i) + ": content plus question " +
                                                   std::to_string(j) + " do not fit the token budget");
                units.push_back(std::move(u));
            }
        }
        int32_t n_user_q = q_base[n_inputs];
        plan->user_q_floor.assign(n_user_q, -1);
        if (o.floors) {
            std::unordered_map<uint64_t, int32_t> first_of_hash;   // hash -> first floor with it
            std::vector<int32_t> next_of_hash;                     // floor -> next floor with its hash
            std::vector<const spinf_question*> floor_q;            // floor -> its question
            for (int32_t i = 0; i < n_inputs; ++i)
                for (int32_t j = 0; j < inputs[i].n_questions; ++j) {
                    const spinf_question& q = inputs[i].questions[j];
                    if (q.kind == SPINF_Q_SEARCHED) continue;   // floors belong to scored questions
                    const uint64_t h = question_hash(q);
                    auto it = first_of_hash.find(h);
                    int32_t f = it == first_of_hash.end() ? -1 : it->second;
                    while (f >= 0 && !same_question(*floor_q[f], q)) f = next_of_hash[f];
                    if (f >= 0) {
                        plan->user_q_floor[q_base[i] + j] = f;
                        continue;
                    }
                    f = (int32_t)floor_q.size();
                    floor_q.push_back(&q);
                    if (it == first_of_hash.end()) {
                        first_of_hash.emplace(h, f);
                        next_of_hash.push_back(-1);
                    } else {   // prepend to the hash's chain (the order of a chain does not matter)
                        next_of_hash.push_back(it->second);
                        it->second = f;
                    }
                    plan->user_q_floor[q_base[i] + j] = f;
                    int64_t size = (int64_t)o.floor_prefix.n + qsize[i][j];
                    if (size > o.token_budget) return fail(SPINF_E_LIMIT, "a floor input does not fit the token budget");
                    Unit u{-1, f, o.floor_prefix, {&q}, {&tries[i][j]}, {f}, size};
                    units.push_back(std::move(u));
                }
        }

        // per-question option bookkeeping for collect
        plan->user_q.assign(n_user_q, QuestionSite{});
        int32_t n_floors = 0;
        for (const Unit& u : units) if (u.source < 0) ++n_floors;
        plan->floor_q.assign(n_floors, QuestionSite{});
        {
            int32_t opt0 = 0;
            for (int32_t i = 0; i < n_inputs; ++i)
                for (int32_t j = 0; j < inputs[i].n_questions; ++j) {
                    const spinf_question& q = inputs[i].questions[j];
                    QuestionSite& s = plan->user_q[q_base[i] + j];
                    s.opt0 = opt0;
                    s.n_options = q.n_options;
                    if (q.kind == SPINF_Q_SEARCHED) ++plan->n_extract;
                    for (int32_t a = 0; a < q.n_options; ++a) plan->opt_len.push_back(q.options[a].n);
                    opt0 += q.n_options;
                }
            plan->n_options_total = opt0;
            plan->extract_k = o.extract_k;
            for (int32_t qi = 0; qi < n_user_q; ++qi) {
                int32_t f = plan->user_q_floor[qi];
                if (f >= 0) {
                    plan->floor_q[f].opt0 = plan->user_q[qi].opt0;
                    plan->floor_q[f].n_options = plan->user_q[qi].n_options;
                }
            }
        }

        // ---- next-fit packing
        std::vector<std::vector<const Unit*>> packs;
        {
            int64_t total = 0;
            for (const Unit& u : units) {
                if (!packs.empty() && !packs.back().empty() && total + u.size > o.token_budget) {
                    packs.emplace_back();
                    total = 0;
                }
                if (packs.empty()) packs.emplace_back();
                packs.back().push_back(&u);
                total += u.size;
            }
        }

        // ---- layout of each pass
        plan->passes.resize(packs.size());
        for (size_t p = 0; p < packs.size(); ++p) {
            Pass& P = plan->passes[p];
            int64_t T64 = 0;
            for (const Unit* u : packs[p]) T64 += u->size;
            const int32_t T = (int32_t)T64;
            const int32_t T_pad = (T + kTile - 1) / kTile * kTile;
            P.T = T;
            P.T_pad = T_pad;
            P.tok.assign(T_pad, 0);
            P.parent.assign(T_pad, -1);
            P.pos.assign(T_pad, 0);
            P.end.resize(T_pad);
            P.anchor.resize(T_pad);
            std::vector<int32_t> g_row;   // packed row of each gather entry
            std::vector<int32_t> x_row;   // packed row of each searched slot
            int32_t r = 0;
            for (const Unit* u : packs[p]) {
                const int32_t s = r, e = r + (int32_t)u->size, L = u->content.n;
                P.unit_start.push_back(s);
                P.unit_source.push_back(u->source);
                for (int32_t i = 0; i < L; ++i, ++r) {
                    P.tok[r] = u->content.ids[i];
                    P.parent[r] = i ? r - 1 : -1;
                    P.pos[r] = i;
                    P.end[r] = e;   // every later row of the input sees the whole content prefix
                    P.anchor[r] = s;
                }
                for (size_t qn = 0; qn < u->qs.size(); ++qn) {
                    const spinf_question& q = *u->qs[qn];
                    const Trie& t = *u->tries[qn];
                    const int32_t qb = r;                                  // first template row
                    const int32_t qe = qb + q.tmpl.n + (int32_t)t.order.size();  // question block end
                    for (int32_t j = 0; j < q.tmpl.n; ++j, ++r) {
                        P.tok[r] = q.tmpl.ids[j];
                        P.parent[r] = j ? r - 1 : (L ? s + L - 1 : -1);
                        P.pos[r] = L + j;
                        P.end[r] = qe;  // later template rows and the whole trie descend from it
                        P.anchor[r] = s;
                    }
                    const int32_t slot = r - 1;
                    if (q.kind == SPINF_Q_SEARCHED) {
                        QuestionSite& dst = plan->user_q[u->qidx[qn]];   // floors hold scored questions only
                        dst.pass = (int32_t)p;
                        dst.x = (int32_t)x_row.size();
                        x_row.push_back(slot);
                        P.x_set.push_back(q.token_set);
                        continue;
                    }
                    const int32_t node0 = r;
                    for (int32_t n : t.order) {
                        P.tok[r] = t.tok[n];
                        P.anchor[r] = s;
                        P.pos[r] = L + q.tmpl.n - 1 + t.depth[n];
                        P.end[r] = r + t.subtree[n];
                        ++r;
                    }
                    for (int32_t c : t.root_kids) P.parent[node0 + t.rank[c]] = slot;
                    for (size_t n = 0; n < t.tok.size(); ++n)
                        for (int32_t c : t.kids[n]) P.parent[node0 + t.rank[c]] = node0 + t.rank[n];
                    QuestionSite site;
                    site.pass = (int32_t)p;
                    site.g0 = (int32_t)g_row.size();
                    for (int32_t a = 0; a < q.n_options; ++a) {
                        const spinf_tokens& opt = q.options[a];
                        for (int32_t i = 0; i < opt.n; ++i) {
                            g_row.push_back(i == 0 ? slot : node0 + t.rank[t.opt_node[a][i]]);
                            P.gather_tok.push_back(opt.ids[i]);
                        }
                    }
                    if (u->source >= 0) {
                        QuestionSite& dst = plan->user_q[u->qidx[qn]];
                        dst.pass = site.pass;
                        dst.g0 = site.g0;
                    } else {
                        QuestionSite& dst = plan->floor_q[u->floor_id];
                        dst.pass = site.pass;
                        dst.g0 = site.g0;
                    }
                }
                if (r != e) return fail(SPINF_E_INVALID, "internal layout size mismatch");
            }
            P.unit_start.push_back(T);
            for (int32_t q = T; q < T_pad; ++q) {
                P.end[q] = q + 1;
                P.anchor[q] = q;
            }

            // Each row's visible keys (its root path) as at most four runs of consecutive
            // rows [lo, hi), for the attention kernel's per-row mask; a row whose path has
            // more runs gets lo0 = -1 and is masked key by key from end[] instead.
            {
                std::vector<int32_t> run_start(T_pad);
                for (int32_t r = 0; r < T_pad; ++r)
                    run_start[r] = (r > 0 && r < T && P.parent[r] == r - 1) ? run_start[r - 1] : r;
                P.row_runs.assign(8 * (size_t)T_pad, 0);
                for (int32_t q = 0; q < T_pad; ++q) {
                    int32_t* out = &P.row_runs[8 * (size_t)q];
                    int32_t hi = q + 1, r = q, n = 0;
                    while (r >= 0) {
                        if (n == 4) {
                            out[0] = -1;
                            break;
                        }
                        const int32_t lo = run_start[r];
                        out[2 * n] = lo;
                        out[2 * n + 1] = hi;
                        ++n;
                        r = lo < T ? P.parent[lo] : -1;
                        hi = r + 1;
                    }
                }
            }

            // KV-tile schedule: per Q tile, per intersecting unit, tiles anchored
            // at the unit start with some key k and some row q of the tile where
            // k <= q < end[k]
            const int32_t n_qt = T_pad / kTile;
            P.tile_ptr.assign(1, 0);
            size_t ub = 0;
            const size_t n_units = packs[p].size();
            for (int32_t qt = 0; qt < n_qt; ++qt) {
                const int32_t r0 = qt * kTile, r1 = r0 + kTile;
                while (ub < n_units && P.unit_start[ub + 1] <= r0) ++ub;
                for (size_t ui = ub; ui < n_units && P.unit_start[ui] < r1; ++ui) {
                    const int32_t s = P.unit_start[ui], e = P.unit_start[ui + 1];
                    const int32_t lo = std::max(r0, s), hi = std::min(r1, e);
                    if (lo >= hi) continue;
                    for (int32_t kb = s; kb < e && kb < hi; kb += kTile) {
                        const int32_t ke = std::min(kb + kTile, e);
                        bool any = false;
                        for (int32_t k = kb; k < ke && !any; ++k)
                            any = std::max(k, lo) < std::min(P.end[k], hi);
                        if (any) {
                            P.tile_kv.push_back(kb);
                            P.tile_len.push_back(ke - kb);
                        }
                    }
                }
                P.tile_ptr.push_back((int32_t)P.tile_kv.size());
            }
            // attention work order: Q tiles with the most KV tiles first (ties: ascending
            // tile), so the persistent CTAs end close together; results do not depend on
            // it.  One 16-byte record {qt, first schedule entry, entry count, 0} per tile.
            std::vector<int32_t> order(n_qt);
            for (int32_t qt = 0; qt < n_qt; ++qt) order[qt] = qt;
            std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
                return P.tile_ptr[a + 1] - P.tile_ptr[a] > P.tile_ptr[b + 1] - P.tile_ptr[b];
            });
            P.qt_work.assign(4 * (size_t)n_qt, 0);
            for (int32_t i = 0; i < n_qt; ++i) {
                const int32_t qt = order[i];
                P.qt_work[4 * i] = qt;
                P.qt_work[4 * i + 1] = P.tile_ptr[qt];
                P.qt_work[4 * i + 2] = P.tile_ptr[qt + 1] - P.tile_ptr[qt];
            }

            // scoring rows: the distinct gather and searched-slot rows, ascending
            std::vector<int32_t> m_of(T > 0 ? T : 1, -1);
            for (int32_t row : g_row) m_of[row] = 0;
            for (int32_t row : x_row) m_of[row] = 0;
            for (int32_t row = 0; row < T; ++row)
                if (m_of[row] >= 0) {
                    m_of[row] = (int32_t)P.slot_row.size();
                    P.slot_row.push_back(row);
                }
            const int32_t G = (int32_t)g_row.size(), M = (int32_t)P.slot_row.size();
            P.gather_m.resize(G);
            for (int32_t g = 0; g < G; ++g) P.gather_m[g] = m_of[g_row[g]];
            P.row_x.assign(M, -1);
            for (size_t x = 0; x < x_row.size(); ++x) {
                P.x_m.push_back(m_of[x_row[x]]);
                P.row_x[m_of[x_row[x]]] = (int32_t)x;
            }
            P.row_gptr.assign(M + 1, 0);
            for (int32_t g = 0; g < G; ++g) P.row_gptr[P.gather_m[g] + 1]++;
            for (int32_t m = 0; m < M; ++m) P.row_gptr[m + 1] += P.row_gptr[m];
            P.row_glist.resize(G);
            {
                std::vector<int32_t> fill(P.row_gptr.begin(), P.row_gptr.end() - 1);
                for (int32_t g = 0; g < G; ++g) P.row_glist[fill[P.gather_m[g]]++] = g;
                for (int32_t m = 0; m < M; ++m)
                    std::sort(P.row_glist.begin() + P.row_gptr[m], P.row_glist.begin() + P.row_gptr[m + 1],
                              [&](int32_t a, int32_t b) {
                                  return P.gather_tok[a] != P.gather_tok[b] ? P.gather_tok[a] < P.gather_tok[b] : a < b;
                              });
            }
        }
        *out = plan.release();
        return SPINF_OK;
    } catch (const std::bad_alloc&) {
        return fail(SPINF_E_NOMEM, "host allocation failed");
    }
}

extern "C" int32_t spinf_plan_num_passes(const spinf_plan* plan) {
    return plan ? (int32_t)plan->passes.size() : 0;
}

extern "C" spinf_status spinf_plan_window_schedule(const spinf_plan* plan, int32_t pass, int32_t window,
                                                   const int32_t** tile_ptr, const int32_t** tile_kv,
                                                   const int32_t** tile_len, int32_t* n_sched) {
    if (!plan || pass < 0 || pass >= (int32_t)plan->passes.size()) return fail(SPINF_E_INVALID, "bad plan or pass");
    if (window <= 0) return fail(SPINF_E_INVALID, "window must be positive");
    if (!tile_ptr || !tile_kv || !tile_len || !n_sched) return fail(SPINF_E_INVALID, "NULL output");
    std::lock_guard<std::mutex> lock(const_cast<spinf_plan*>(plan)->cache_mu);
    WindowSchedule& w = window_schedule(const_cast<Pass&>(plan->passes[pass]), window);
    *tile_ptr = w.tile_ptr.data();
    *tile_kv = w.tile_kv.data();
    *tile_len = w.tile_len.data();
    *n_sched = (int32_t)w.tile_kv.size();
    return SPINF_OK;
}

extern "C" spinf_status spinf_plan_tile_schedule(const spinf_plan* plan, int32_t pass, int32_t window,
                                                 int32_t key_tile, const int32_t** tile_ptr, const int32_t** tile_kv,
                                                 const int32_t** tile_len, int32_t* n_sched) {
    return spinf_plan_tile_schedule_q(plan, pass, window, key_tile, kTile, tile_ptr, tile_kv, tile_len, n_sched);
}

extern "C" spinf_status spinf_plan_tile_schedule_q(const spinf_plan* plan, int32_t pass, int32_t window,
                                                   int32_t key_tile, int32_t q_rows, const int32_t** tile_ptr,
                                                   const int32_t** tile_kv, const int32_t** tile_len,
                                                   int32_t* n_sched) {
    if (!plan || pass < 0 || pass >= (int32_t)plan->passes.size()) return fail(SPINF_E_INVALID, "bad plan or pass");
    if (window < 0) return fail(SPINF_E_INVALID, "negative window");
    if (key_tile != 64 && key_tile != kTile) return fail(SPINF_E_INVALID, "key_tile must be 64 or 128");
    if (q_rows != 64 && q_rows != kTile) return fail(SPINF_E_INVALID, "q_rows must be 64 or 128");
    if (!tile_ptr || !tile_kv || !tile_len || !n_sched) return fail(SPINF_E_INVALID, "NULL output");
    std::lock_guard<std::mutex> lock(const_cast<spinf_plan*>(plan)->cache_mu);
    WindowSchedule& w = tile_schedule(const_cast<Pass&>(plan->passes[pass]), window, key_tile, q_rows);
    *tile_ptr = w.tile_ptr.data();
    *tile_kv = w.tile_kv.data();
    *tile_len = w.tile_len.data();
    *n_sched = (int32_t)w.tile_kv.size();
    return SPINF_OK;
}

extern "C" spinf_status spinf_plan_pass_info(const spinf_plan* plan, int32_t pass, spinf_pass_info* out) {
    if (!plan || !out || pass < 0 || pass >= (int32_t)plan->passes.size())
        return fail(SPINF_E_INVALID, "bad plan or pass index");
    const Pass& P = plan->passes[pass];
    out->T = P.T;
    out->T_pad = P.T_pad;
    out->n_qtiles = P.T_pad / kTile;
    out->n_sched = (int32_t)P.tile_kv.size();
    out->M = (int32_t)P.slot_row.size();
    out->G = (int32_t)P.gather_tok.size();
    out->n_units = (int32_t)P.unit_source.size();
    out->tok = P.tok.data();
    out->parent = P.parent.data();
    out->pos = P.pos.data();
    out->end = P.end.data();
    out->anchor = P.anchor.data();
    out->tile_ptr = P.tile_ptr.data();
    out->tile_kv = P.tile_kv.data();
    out->tile_len = P.tile_len.data();
    out->slot_row = P.slot_row.data();
    out->gather_m = P.gather_m.data();
    out->gather_tok = P.gather_tok.data();
    out->unit_start = P.unit_start.data();
    out->unit_source = P.unit_source.data();
    out->row_runs = P.row_runs.data();
    out->X = (int32_t)P.x_m.size();
    out->x_m = P.x_m.data();
    out->x_set = P.x_set.data();
    return SPINF_OK;
}

extern "C" spinf_status spinf_plan_counts(const spinf_plan* plan, int64_t* n_questions, int64_t* n_options) {
    if (!plan) return fail(SPINF_E_INVALID, "plan is NULL");
    if (n_questions) *n_questions = (int64_t)plan->user_q.size();
    if (n_options) *n_options = plan->n_options_total;
    return SPINF_OK;
}

extern "C" spinf_status spinf_plan_extract_counts(const spinf_plan* plan, int64_t* n_extract, int32_t* extract_k) {
    if (!plan) return fail(SPINF_E_INVALID, "plan is NULL");
    if (n_extract) *n_extract = plan->n_extract;
    if (extract_k) *extract_k = plan->extract_k;
    return SPINF_OK;
}

namespace {

// lp per option of one laid-out question, then p and residual, in fp64
void question_stats(const spinf_plan* plan, const QuestionSite& s, const float* tlp, double* lp, double* p,
                    double* residual) {
    int32_t g = s.g0;
    double m = -INFINITY;
    for (int32_t a = 0; a < s.n_options; ++a) {
        double acc = 0.0;
        for (int32_t i = 0; i < plan->opt_len[s.opt0 + a]; ++i) acc += (double)tlp[g++];
        lp[a] = acc;
        m = std::max(m, acc);
    }
    double sum = 0.0;
    for (int32_t a = 0; a < s.n_options; ++a) {
        p[a] = std::exp(lp[a] - m);
        sum += p[a];
    }
    for (int32_t a = 0; a < s.n_options; ++a) p[a] /= sum;
    *residual = -std::expm1(m + std::log(sum));
}

}  // namespace

extern "C" spinf_status spinf_collect(const spinf_plan* plan, const float* const* tlp, const spinf_result* out) {
    if (!plan || !out) return fail(SPINF_E_INVALID, "plan or result is NULL");
    if (!plan->passes.empty() && !tlp) return fail(SPINF_E_INVALID, "token log-probabilities are NULL");
    for (size_t p = 0; p < plan->passes.size(); ++p)
        if (!tlp[p] && !plan->passes[p].gather_tok.empty())
            return fail(SPINF_E_INVALID, "token log-probabilities of a pass are NULL");
    if (!out->option_lp || !out->option_p || !out->residual)
        return fail(SPINF_E_INVALID, "result arrays are NULL");
    // each floor once: many user questions share one
    const size_t n_floors = plan->floor_q.size();
    std::vector<size_t> foff(n_floors + 1, 0);
    for (size_t f = 0; f < n_floors; ++f) foff[f + 1] = foff[f] + plan->floor_q[f].n_options;
    std::vector<double> flp(foff.back()), fp(foff.back()), fres(n_floors);
    for (size_t f = 0; f < n_floors; ++f) {
        const QuestionSite& fs = plan->floor_q[f];
        question_stats(plan, fs, tlp[fs.pass], flp.data() + foff[f], fp.data() + foff[f], &fres[f]);
    }
    for (size_t qi = 0; qi < plan->user_q.size(); ++qi) {
        const QuestionSite& s = plan->user_q[qi];
        if (s.x >= 0) {   // a searched slot: no options, no floor
            out->residual[qi] = NAN;
            if (out->floor_residual) out->floor_residual[qi] = NAN;
            continue;
        }
        question_stats(plan, s, tlp[s.pass], out->option_lp + s.opt0, out->option_p + s.opt0, out->residual + qi);
        const int32_t f = plan->user_q_floor[qi];
        for (int32_t a = 0; a < s.n_options; ++a) {
            if (out->option_floor_lp) out->option_floor_lp[s.opt0 + a] = f >= 0 ? flp[foff[f] + a] : NAN;
            if (out->option_floor_p) out->option_floor_p[s.opt0 + a] = f >= 0 ? fp[foff[f] + a] : NAN;
        }
        if (out->floor_residual) out->floor_residual[qi] = f >= 0 ? fres[f] : NAN;
    }
    return SPINF_OK;
}

extern "C" spinf_status spinf_collect_extract(const spinf_plan* plan, const int32_t* const* top_tok,
                                              const float* const* top_lp, int32_t* tok, double* lp) {
    if (!plan) return fail(SPINF_E_INVALID, "plan is NULL");
    if (plan->n_extract == 0) return SPINF_OK;
    if (!top_tok || !top_lp || !tok || !lp) return fail(SPINF_E_INVALID, "NULL arrays");
    const int32_t k = plan->extract_k;
    int64_t e = 0;
    for (const QuestionSite& s : plan->user_q) {
        if (s.x < 0) continue;
        const int32_t* st = top_tok[s.pass];
        const float* sl = top_lp[s.pass];
        if (!st || !sl) return fail(SPINF_E_INVALID, "answers of a pass are NULL");
        for (int32_t j = 0; j < k; ++j) {
            tok[e * k + j] = st[(size_t)s.x * k + j];
            lp[e * k + j] = (double)sl[(size_t)s.x * k + j];
        }
        ++e;
    }
    return SPINF_OK;
}

extern "C" const char* spinf_status_string(spinf_status s) {
    switch (s) {
        case SPINF_OK: return "ok";
        case SPINF_E_INVALID: return "invalid argument";
        case SPINF_E_LIMIT: return "limit exceeded";
        case SPINF_E_NOMEM: return "out of memory";
        case SPINF_E_CUDA: return "CUDA error";
        case SPINF_E_UNSUPPORTED: return "unsupported";
        case SPINF_E_DEVICE_TIMEOUT: return "device wait timed out";
        case SPINF_E_DEVICE_CHECK: return "device check failed";
    }
    return "unknown status";
}

extern "C" const char* spinf_last_error(void) { return g_last_error.c_str(); }
