// layout.cpp -- GF(2) linear layouts (host).
//
// A layout is a linear map over GF(2) from named input dims (register, lane,
// warp, thread, offset, ...) to named output dims (tensor coordinates), kept
// as one basis vector per input bit with one coordinate per output dim
// (retepy.com "Triton LinearLayout", sections "Linear Layout" and
// "Basis-vector representation").  Evaluation XORs the bases of the set input
// bits ("LinearLayout::apply"); composition applies the outer layout to every
// basis ("Combining layouts"); rank comes from row reduction over GF(2), and
// injectivity / surjectivity compare it with the input / output bit counts
// ("Surjectivity, injectivity, and broadcasts"); invertAndCompose solves a
// GF(2) linear system with free variables set to zero ("invertAndCompose").
//
// The constructors describe the ownership maps this library uses or the
// pages define: the rank-2 blocked encoding, cooperative tile traversal and
// strided register tiles of the mytriton pages, the 128-byte shared-memory
// swizzle the TMA writes and the tensor cores read, and the tcgen05.ld 32x32b
// accumulator readout.
#include <cstdint>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "../../include/tilegemm.h"

struct tg_layout {
    std::vector<std::string> in_names;
    std::vector<int> in_bits;
    std::vector<std::string> out_names;
    std::vector<int> out_bits;
    std::vector<std::vector<int32_t>> bases;  // [total in bits][n_out]
};

namespace {

struct LayoutError {};

int total(const std::vector<int>& bits) {
    int t = 0;
    for (int b : bits) t += b;
    return t;
}

int find(const std::vector<std::string>& names, const std::string& n) {
    for (size_t i = 0; i < names.size(); ++i)
        if (names[i] == n) return (int)i;
    return -1;
}

int offset_of(const std::vector<int>& bits, int dim) {
    int o = 0;
    for (int i = 0; i < dim; ++i) o += bits[i];
    return o;
}

void check(const tg_layout& l) {
    auto names_ok = [](const std::vector<std::string>& names, const std::vector<int>& bits) {
        if (names.size() != bits.size()) return false;
        for (size_t i = 0; i < names.size(); ++i) {
            if (names[i].empty() || names[i].size() > 31) return false;
            if (bits[i] < 0 || bits[i] > 30) return false;
            for (size_t j = 0; j < i; ++j)
                if (names[j] == names[i]) return false;
        }
        return true;
    };
    if (!names_ok(l.in_names, l.in_bits) || !names_ok(l.out_names, l.out_bits)) throw LayoutError();
    if (total(l.in_bits) > 63 || total(l.out_bits) > 63) throw LayoutError();
    if ((int)l.bases.size() != total(l.in_bits)) throw LayoutError();
    for (const auto& b : l.bases) {
        if (b.size() != l.out_names.size()) throw LayoutError();
        for (size_t o = 0; o < b.size(); ++o)
            if (b[o] < 0 || b[o] >= (1 << l.out_bits[o])) throw LayoutError();
    }
}

std::vector<int32_t> apply(const tg_layout& l, const int32_t* ins) {
    std::vector<int32_t> out(l.out_names.size(), 0);
    int row = 0;
    for (size_t d = 0; d < l.in_names.size(); ++d) {
        for (int i = 0; i < l.in_bits[d]; ++i, ++row) {
            if (ins[d] & (1 << i))
                for (size_t o = 0; o < out.size(); ++o) out[o] ^= l.bases[row][o];
        }
    }
    return out;
}

// Output coordinates flattened into one bit vector (first out dim lowest).
uint64_t flatten(const tg_layout& l, const std::vector<int32_t>& coords) {
    uint64_t v = 0;
    int shift = 0;
    for (size_t o = 0; o < coords.size(); ++o) {
        v |= (uint64_t)(uint32_t)coords[o] << shift;
        shift += l.out_bits[o];
    }
    return v;
}

// Row reduction over GF(2): pivots indexed by leading bit, each carrying the
// combination of input columns that produced it.
struct Echelon {
    uint64_t vec[64] = {};
    uint64_t comb[64] = {};
    bool has[64] = {};
    int rank = 0;

    void insert(uint64_t v, uint64_t c) {
        for (int b = 63; b >= 0; --b) {
            if (!((v >> b) & 1)) continue;
            if (has[b]) {
                v ^= vec[b];
                c ^= comb[b];
            } else {
                vec[b] = v;
                comb[b] = c;
                has[b] = true;
                ++rank;
                return;
            }
        }
    }

    // Combination of columns whose XOR is t (free columns get 0); false if t
    // is outside the span.
    bool solve(uint64_t t, uint64_t* x) const {
        uint64_t c = 0;
        for (int b = 63; b >= 0; --b) {
            if (!((t >> b) & 1)) continue;
            if (!has[b]) return false;
            t ^= vec[b];
            c ^= comb[b];
        }
        *x = c;
        return true;
    }
};

Echelon reduce(const tg_layout& l) {
    Echelon e;
    for (size_t r = 0; r < l.bases.size(); ++r) e.insert(flatten(l, l.bases[r]), 1ull << r);
    return e;
}

int log2_exact(int v) {
    if (v <= 0 || (v & (v - 1))) throw LayoutError();
    int b = 0;
    while ((1 << b) < v) ++b;
    return b;
}

tg_layout* make(std::vector<std::string> in_names, std::vector<int> in_bits,
                std::vector<std::string> out_names, std::vector<int> out_bits) {
    tg_layout* l = new tg_layout;
    l->in_names = std::move(in_names);
    l->in_bits = std::move(in_bits);
    l->out_names = std::move(out_names);
    l->out_bits = std::move(out_bits);
    return l;
}

template <class F>
int guarded(F&& f) {
    try {
        return f();
    } catch (const LayoutError&) {
        return TG_ERR_LAYOUT;
    } catch (const std::bad_alloc&) {
        return TG_ERR_LAYOUT;
    }
}

std::vector<std::string> names_of(int n, const char* const* names) {
    if (n < 0 || (n > 0 && !names)) throw LayoutError();
    std::vector<std::string> v;
    for (int i = 0; i < n; ++i) {
        if (!names[i]) throw LayoutError();
        v.emplace_back(names[i]);
    }
    return v;
}

int copy_name(const std::string& s, char* name, size_t len) {
    if (!name) return TG_OK;
    if (s.size() + 1 > len) return TG_ERR_BUFFER;
    std::memcpy(name, s.c_str(), s.size() + 1);
    return TG_OK;
}

}  // namespace

extern "C" {

int tg_layout_create(int n_in, const char* const* in_names, const int* in_bits, int n_out,
                     const char* const* out_names, const int* out_bits, const int32_t* bases,
                     tg_layout** out) {
    if (!out || (n_in > 0 && !in_bits) || (n_out > 0 && !out_bits)) return TG_ERR_INVALID_ARG;
    return guarded([&] {
        std::vector<int> ib(in_bits, in_bits + (n_in > 0 ? n_in : 0));
        std::vector<int> ob(out_bits, out_bits + (n_out > 0 ? n_out : 0));
        tg_layout* l = make(names_of(n_in, in_names), ib, names_of(n_out, out_names), ob);
        const int rows = total(ib) > 63 ? -1 : total(ib);
        if (rows < 0 || (rows > 0 && n_out > 0 && !bases)) {
            delete l;
            throw LayoutError();
        }
        for (int r = 0; r < rows; ++r)
            l->bases.emplace_back(bases + (size_t)r * n_out, bases + (size_t)(r + 1) * n_out);
        try {
            check(*l);
        } catch (...) {
            delete l;
            throw;
        }
        *out = l;
        return TG_OK;
    });
}

void tg_layout_destroy(tg_layout* l) { delete l; }

int tg_layout_num_dims(const tg_layout* l, int* n_in, int* n_out) {
    if (!l) return TG_ERR_INVALID_ARG;
    if (n_in) *n_in = (int)l->in_names.size();
    if (n_out) *n_out = (int)l->out_names.size();
    return TG_OK;
}

int tg_layout_in_dim(const tg_layout* l, int i, char* name, size_t len, int* bits) {
    if (!l || i < 0 || i >= (int)l->in_names.size()) return TG_ERR_INVALID_ARG;
    if (bits) *bits = l->in_bits[i];
    return copy_name(l->in_names[i], name, len);
}

int tg_layout_out_dim(const tg_layout* l, int i, char* name, size_t len, int* bits) {
    if (!l || i < 0 || i >= (int)l->out_names.size()) return TG_ERR_INVALID_ARG;
    if (bits) *bits = l->out_bits[i];
    return copy_name(l->out_names[i], name, len);
}

int tg_layout_get_bases(const tg_layout* l, int32_t* bases, size_t count) {
    if (!l) return TG_ERR_INVALID_ARG;
    const size_t need = l->bases.size() * l->out_names.size();
    if (count < need) return TG_ERR_BUFFER;
    if (need && !bases) return TG_ERR_INVALID_ARG;
    size_t k = 0;
    for (const auto& b : l->bases)
        for (int32_t v : b) bases[k++] = v;
    return TG_OK;
}

int tg_layout_apply(const tg_layout* l, const int32_t* ins, int32_t* outs) {
    if (!l || (!ins && !l->in_names.empty()) || (!outs && !l->out_names.empty()))
        return TG_ERR_INVALID_ARG;
    for (size_t d = 0; d < l->in_names.size(); ++d)
        if (ins[d] < 0 || ins[d] >= (1 << l->in_bits[d])) return TG_ERR_INVALID_ARG;
    const std::vector<int32_t> o = apply(*l, ins);
    for (size_t i = 0; i < o.size(); ++i) outs[i] = o[i];
    return TG_OK;
}

int tg_layout_compose(const tg_layout* inner, const tg_layout* outer, tg_layout** out) {
    if (!inner || !outer || !out) return TG_ERR_INVALID_ARG;
    return guarded([&] {
        if (inner->out_names != outer->in_names || inner->out_bits != outer->in_bits)
            throw LayoutError();
        tg_layout* l = make(inner->in_names, inner->in_bits, outer->out_names, outer->out_bits);
        for (const auto& b : inner->bases) l->bases.push_back(apply(*outer, b.data()));
        *out = l;
        return TG_OK;
    });
}

int tg_layout_product(const tg_layout* a, const tg_layout* b, tg_layout** out) {
    if (!a || !b || !out) return TG_ERR_INVALID_ARG;
    return guarded([&] {
        std::vector<std::string> in_names = a->in_names, out_names = a->out_names;
        std::vector<int> in_bits = a->in_bits, out_bits = a->out_bits;
        for (size_t d = 0; d < b->in_names.size(); ++d) {
            const int k = find(in_names, b->in_names[d]);
            if (k < 0) {
                in_names.push_back(b->in_names[d]);
                in_bits.push_back(b->in_bits[d]);
            } else {
                in_bits[k] += b->in_bits[d];
            }
        }
        for (size_t o = 0; o < b->out_names.size(); ++o) {
            const int k = find(out_names, b->out_names[o]);
            if (k < 0) {
                out_names.push_back(b->out_names[o]);
                out_bits.push_back(b->out_bits[o]);
            } else {
                out_bits[k] += b->out_bits[o];
            }
        }
        tg_layout* l = make(in_names, in_bits, out_names, out_bits);
        for (size_t d = 0; d < in_names.size(); ++d) {
            const int da = find(a->in_names, in_names[d]);
            const int db = find(b->in_names, in_names[d]);
            if (da >= 0) {  // a's bits first (least significant)
                const int base = offset_of(a->in_bits, da);
                for (int i = 0; i < a->in_bits[da]; ++i) {
                    std::vector<int32_t> v(out_names.size(), 0);
                    for (size_t o = 0; o < a->out_names.size(); ++o)
                        v[find(out_names, a->out_names[o])] = a->bases[base + i][o];
                    l->bases.push_back(v);
                }
            }
            if (db >= 0) {  // then b's, whose shared output coordinates move up
                const int base = offset_of(b->in_bits, db);
                for (int i = 0; i < b->in_bits[db]; ++i) {
                    std::vector<int32_t> v(out_names.size(), 0);
                    for (size_t o = 0; o < b->out_names.size(); ++o) {
                        const int ao = find(a->out_names, b->out_names[o]);
                        const int shift = ao >= 0 ? a->out_bits[ao] : 0;
                        v[find(out_names, b->out_names[o])] = b->bases[base + i][o] << shift;
                    }
                    l->bases.push_back(v);
                }
            }
        }
        try {
            check(*l);
        } catch (...) {
            delete l;
            throw;
        }
        *out = l;
        return TG_OK;
    });
}

int tg_layout_sublayout(const tg_layout* l, int n_in, const char* const* in_names, int n_out,
                        const char* const* out_names, tg_layout** out) {
    if (!l || !out) return TG_ERR_INVALID_ARG;
    return guarded([&] {
        const std::vector<std::string> ins = names_of(n_in, in_names), outs = names_of(n_out, out_names);
        std::vector<int> ib, ob, oi;
        for (const auto& n : ins) {
            const int d = find(l->in_names, n);
            if (d < 0) throw LayoutError();
            ib.push_back(l->in_bits[d]);
        }
        for (const auto& n : outs) {
            const int o = find(l->out_names, n);
            if (o < 0) throw LayoutError();
            ob.push_back(l->out_bits[o]);
            oi.push_back(o);
        }
        tg_layout* r = make(ins, ib, outs, ob);
        for (const auto& n : ins) {
            const int d = find(l->in_names, n);
            const int base = offset_of(l->in_bits, d);
            for (int i = 0; i < l->in_bits[d]; ++i) {
                std::vector<int32_t> v;
                for (int o : oi) v.push_back(l->bases[base + i][o]);
                r->bases.push_back(v);
            }
        }
        try {
            check(*r);
        } catch (...) {
            delete r;
            throw;
        }
        *out = r;
        return TG_OK;
    });
}

int tg_layout_transpose_outs(const tg_layout* l, int n_out, const char* const* out_names,
                             tg_layout** out) {
    if (!l || !out) return TG_ERR_INVALID_ARG;
    if (n_out != (int)l->out_names.size()) return TG_ERR_LAYOUT;
    std::vector<const char*> ins;
    for (const auto& n : l->in_names) ins.push_back(n.c_str());
    return tg_layout_sublayout(l, (int)ins.size(), ins.data(), n_out, out_names, out);
}

int tg_layout_transpose_ins(const tg_layout* l, int n_in, const char* const* in_names,
                            tg_layout** out) {
    if (!l || !out) return TG_ERR_INVALID_ARG;
    if (n_in != (int)l->in_names.size()) return TG_ERR_LAYOUT;
    std::vector<const char*> outs;
    for (const auto& n : l->out_names) outs.push_back(n.c_str());
    return tg_layout_sublayout(l, n_in, in_names, (int)outs.size(), outs.data(), out);
}

int tg_layout_reshape_ins(const tg_layout* l, int n_in, const char* const* in_names,
                          const int* in_bits, tg_layout** out) {
    if (!l || !out || (n_in > 0 && !in_bits)) return TG_ERR_INVALID_ARG;
    return guarded([&] {
        std::vector<int> ib(in_bits, in_bits + (n_in > 0 ? n_in : 0));
        for (int b : ib)
            if (b < 0) throw LayoutError();
        if (total(ib) != total(l->in_bits)) throw LayoutError();
        // the bases stay in flattened order: only the grouping into dims changes
        tg_layout* r = make(names_of(n_in, in_names), ib, l->out_names, l->out_bits);
        r->bases = l->bases;
        try {
            check(*r);
        } catch (...) {
            delete r;
            throw;
        }
        *out = r;
        return TG_OK;
    });
}

int tg_layout_reshape_outs(const tg_layout* l, int n_out, const char* const* out_names,
                           const int* out_bits, tg_layout** out) {
    if (!l || !out || (n_out > 0 && !out_bits)) return TG_ERR_INVALID_ARG;
    return guarded([&] {
        std::vector<int> ob(out_bits, out_bits + (n_out > 0 ? n_out : 0));
        for (int b : ob)
            if (b < 0 || b > 30) throw LayoutError();
        if (total(ob) != total(l->out_bits)) throw LayoutError();
        tg_layout* r = make(l->in_names, l->in_bits, names_of(n_out, out_names), ob);
        for (const auto& b : l->bases) {
            const uint64_t f = flatten(*l, b);  // first out dim lowest
            std::vector<int32_t> v;
            int shift = 0;
            for (int bits : ob) {
                v.push_back((int32_t)((f >> shift) & ((1ull << bits) - 1)));
                shift += bits;
            }
            r->bases.push_back(v);
        }
        try {
            check(*r);
        } catch (...) {
            delete r;
            throw;
        }
        *out = r;
        return TG_OK;
    });
}

}  // extern "C"

namespace {

// Whether P and A are the same map once their dims are matched by name.
bool same_map(const tg_layout& P, const tg_layout& A) {
    if (P.in_names.size() != A.in_names.size() || P.out_names.size() != A.out_names.size())
        return false;
    std::vector<int> out_of_p;  // P's out dim for each of A's
    for (size_t o = 0; o < A.out_names.size(); ++o) {
        const int k = find(P.out_names, A.out_names[o]);
        if (k < 0 || P.out_bits[k] != A.out_bits[o]) return false;
        out_of_p.push_back(k);
    }
    for (size_t d = 0; d < A.in_names.size(); ++d) {
        const int k = find(P.in_names, A.in_names[d]);
        if (k < 0 || P.in_bits[k] != A.in_bits[d]) return false;
        const int pa = offset_of(A.in_bits, (int)d), pp = offset_of(P.in_bits, k);
        for (int i = 0; i < A.in_bits[d]; ++i)
            for (size_t o = 0; o < A.out_names.size(); ++o)
                if (P.bases[pp + i][out_of_p[o]] != A.bases[pa + i][o]) return false;
    }
    return true;
}

// divideLeft (A = B * C) and divideRight (A = C * B) under the product's
// convention that, for a dim both factors have, the left factor owns the low
// input bits and the low output bits.  C keeps A's dims and order, each with
// A's bits less B's.
int divide(const tg_layout* A, const tg_layout* B, bool left, tg_layout** out) {
    if (!A || !B || !out) return TG_ERR_INVALID_ARG;
    return guarded([&] {
        for (const auto& n : B->in_names)
            if (find(A->in_names, n) < 0) throw LayoutError();
        for (const auto& n : B->out_names)
            if (find(A->out_names, n) < 0) throw LayoutError();
        std::vector<int> b_in(A->in_names.size(), 0), c_in, b_out(A->out_names.size(), 0), c_out;
        for (size_t d = 0; d < A->in_names.size(); ++d) {
            const int k = find(B->in_names, A->in_names[d]);
            if (k >= 0) b_in[d] = B->in_bits[k];
            if (b_in[d] > A->in_bits[d]) throw LayoutError();
            c_in.push_back(A->in_bits[d] - b_in[d]);
        }
        for (size_t o = 0; o < A->out_names.size(); ++o) {
            const int k = find(B->out_names, A->out_names[o]);
            if (k >= 0) b_out[o] = B->out_bits[k];
            if (b_out[o] > A->out_bits[o]) throw LayoutError();
            c_out.push_back(A->out_bits[o] - b_out[o]);
        }
        tg_layout* C = make(A->in_names, c_in, A->out_names, c_out);
        try {
            for (size_t d = 0; d < A->in_names.size(); ++d) {
                const int base = offset_of(A->in_bits, (int)d);
                const int first = left ? b_in[d] : 0;  // C's bits of this dim
                for (int i = first; i < first + c_in[d]; ++i) {
                    std::vector<int32_t> v;
                    for (size_t o = 0; o < A->out_names.size(); ++o) {
                        const int32_t c = A->bases[base + i][o];
                        if (left) {  // C's coordinates sit above B's
                            if (c & ((1 << b_out[o]) - 1)) throw LayoutError();
                            v.push_back(c >> b_out[o]);
                        } else {     // C's coordinates sit below B's
                            if (c >> c_out[o]) throw LayoutError();
                            v.push_back(c);
                        }
                    }
                    C->bases.push_back(v);
                }
            }
            check(*C);
            // B's part of A must be B itself: rebuild the product and compare.
            tg_layout* P = nullptr;
            const int rc = left ? tg_layout_product(B, C, &P) : tg_layout_product(C, B, &P);
            if (rc != TG_OK) throw LayoutError();
            const bool same = same_map(*P, *A);
            delete P;
            if (!same) throw LayoutError();
        } catch (...) {
            delete C;
            throw;
        }
        *out = C;
        return TG_OK;
    });
}

}  // namespace

extern "C" {

int tg_layout_divide_left(const tg_layout* A, const tg_layout* B, tg_layout** out) {
    return divide(A, B, true, out);
}

int tg_layout_divide_right(const tg_layout* A, const tg_layout* B, tg_layout** out) {
    return divide(A, B, false, out);
}

int tg_layout_rank(const tg_layout* l, int* value) {
    if (!l || !value) return TG_ERR_INVALID_ARG;
    *value = reduce(*l).rank;
    return TG_OK;
}

int tg_layout_is_injective(const tg_layout* l, int* value) {
    if (!l || !value) return TG_ERR_INVALID_ARG;
    *value = reduce(*l).rank == total(l->in_bits);
    return TG_OK;
}

int tg_layout_is_surjective(const tg_layout* l, int* value) {
    if (!l || !value) return TG_ERR_INVALID_ARG;
    *value = reduce(*l).rank == total(l->out_bits);
    return TG_OK;
}

int tg_layout_invert_and_compose(const tg_layout* R, const tg_layout* S, tg_layout** out) {
    if (!R || !S || !out) return TG_ERR_INVALID_ARG;
    return guarded([&] {
        // S's output dims in R's order (same names and sizes required).
        if (R->out_names.size() != S->out_names.size()) throw LayoutError();
        std::vector<const char*> order;
        for (size_t o = 0; o < R->out_names.size(); ++o) {
            const int k = find(S->out_names, R->out_names[o]);
            if (k < 0 || S->out_bits[k] != R->out_bits[o]) throw LayoutError();
            order.push_back(R->out_names[o].c_str());
        }
        tg_layout* St = nullptr;
        if (tg_layout_transpose_outs(S, (int)order.size(), order.data(), &St) != TG_OK)
            throw LayoutError();
        const Echelon e = reduce(*St);
        delete St;
        tg_layout* l = make(R->in_names, R->in_bits, S->in_names, S->in_bits);
        for (const auto& b : R->bases) {
            uint64_t x = 0;
            if (!e.solve(flatten(*R, b), &x)) {
                delete l;
                throw LayoutError();
            }
            std::vector<int32_t> v(S->in_names.size(), 0);
            int bit = 0;
            for (size_t d = 0; d < S->in_names.size(); ++d)
                for (int i = 0; i < S->in_bits[d]; ++i, ++bit)
                    if ((x >> bit) & 1) v[d] |= 1 << i;
            l->bases.push_back(v);
        }
        *out = l;
        return TG_OK;
    });
}

int tg_layout_blocked_nd(int rank, const int* size_per_thread, const int* threads_per_warp,
                         const int* warps_per_cta, const int* order, const int* shape,
                         tg_layout** out) {
    if (!size_per_thread || !threads_per_warp || !warps_per_cta || !order || !shape || !out ||
        rank < 1 || rank > 8)
        return TG_ERR_INVALID_ARG;
    return guarded([&] {
        std::vector<int> seen(rank, 0);  // `order` is a permutation of 0 .. rank-1
        for (int k = 0; k < rank; ++k) {
            if (order[k] < 0 || order[k] >= rank || seen[order[k]]++) throw LayoutError();
        }
        std::vector<int> lg_spt(rank), lg_tpw(rank), lg_wpc(rank), lg_shape(rank), lg_rep(rank);
        for (int d = 0; d < rank; ++d) {
            lg_spt[d] = log2_exact(size_per_thread[d]);
            lg_tpw[d] = log2_exact(threads_per_warp[d]);
            lg_wpc[d] = log2_exact(warps_per_cta[d]);
            lg_shape[d] = log2_exact(shape[d]);
            const int tile = lg_spt[d] + lg_tpw[d] + lg_wpc[d];
            lg_rep[d] = lg_shape[d] > tile ? lg_shape[d] - tile : 0;
        }
        // Coordinate (1 << lg) along dim d, or a broadcast (zero) basis when
        // the CTA tile is larger than the tensor along d.
        auto basis = [&](int d, int lg) {
            std::vector<int32_t> v(rank, 0);
            if (lg < lg_shape[d]) v[d] = 1 << lg;
            return v;
        };
        std::vector<std::string> out_names;
        for (int d = 0; d < rank; ++d) out_names.push_back("dim" + std::to_string(d));
        tg_layout* l = make({"register", "lane", "warp"}, {0, 0, 0}, out_names, lg_shape);
        // per dim in `order` (minor first): the thread's own elements, then
        // lanes, then warps; then the CTA tile's repetitions as more registers
        std::vector<std::vector<int32_t>> reg, lane, warp;
        for (int k = 0; k < rank; ++k) {
            const int d = order[k];
            for (int i = 0; i < lg_spt[d]; ++i) reg.push_back(basis(d, i));
            for (int i = 0; i < lg_tpw[d]; ++i) lane.push_back(basis(d, lg_spt[d] + i));
            for (int i = 0; i < lg_wpc[d]; ++i) warp.push_back(basis(d, lg_spt[d] + lg_tpw[d] + i));
        }
        for (int k = 0; k < rank; ++k) {
            const int d = order[k];
            for (int i = 0; i < lg_rep[d]; ++i)
                reg.push_back(basis(d, lg_spt[d] + lg_tpw[d] + lg_wpc[d] + i));
        }
        l->in_bits = {(int)reg.size(), (int)lane.size(), (int)warp.size()};
        for (auto* group : {&reg, &lane, &warp})
            for (auto& v : *group) l->bases.push_back(v);
        try {
            check(*l);
        } catch (...) {
            delete l;
            throw;
        }
        *out = l;
        return TG_OK;
    });
}

int tg_layout_blocked(const int size_per_thread[2], const int threads_per_warp[2],
                      const int warps_per_cta[2], const int order[2], const int shape[2],
                      tg_layout** out) {
    return tg_layout_blocked_nd(2, size_per_thread, threads_per_warp, warps_per_cta, order, shape,
                                out);
}

int tg_layout_cooperative(const int shape[2], int threads, const int order[2], tg_layout** out) {
    if (!shape || !order || !out) return TG_ERR_INVALID_ARG;
    return guarded([&] {
        if (!((order[0] == 0 && order[1] == 1) || (order[0] == 1 && order[1] == 0)))
            throw LayoutError();
        const int lg_s0 = log2_exact(shape[0]), lg_s1 = log2_exact(shape[1]);
        const int lg_t = log2_exact(threads);
        const int lg_size = lg_s0 + lg_s1;
        if (lg_t > lg_size || threads > 1024) throw LayoutError();
        tg_layout* l = make({"thread", "iteration"}, {lg_t, lg_size - lg_t}, {"dim0", "dim1"},
                            {lg_s0, lg_s1});
        // linear index t + i*threads; bit b of it lands on the axis peeled at
        // that position (fastest axis first).
        for (int b = 0; b < lg_size; ++b) {
            int64_t rem = 1LL << b;
            std::vector<int32_t> v(2, 0);
            for (int k = 0; k < 2; ++k) {
                const int ax = order[k];
                v[ax] = (int32_t)(rem % shape[ax]);
                rem /= shape[ax];
            }
            l->bases.push_back(v);
        }
        *out = l;
        return TG_OK;
    });
}

int tg_layout_register_tile(const int logical[2], const int thread_shape[2], tg_layout** out) {
    if (!logical || !thread_shape || !out) return TG_ERR_INVALID_ARG;
    return guarded([&] {
        int lg_l[2], lg_t[2], lg_r[2];
        for (int d = 0; d < 2; ++d) {
            lg_l[d] = log2_exact(logical[d]);
            lg_t[d] = log2_exact(thread_shape[d]);
            if (lg_t[d] > lg_l[d]) throw LayoutError();
            lg_r[d] = lg_l[d] - lg_t[d];
        }
        tg_layout* l = make({"register", "thread"}, {lg_r[0] + lg_r[1], lg_t[0] + lg_t[1]},
                            {"dim0", "dim1"}, {lg_l[0], lg_l[1]});
        // register id row-major over the register shape: low bits = column
        for (int i = 0; i < lg_r[1]; ++i) l->bases.push_back({0, thread_shape[1] << i});
        for (int i = 0; i < lg_r[0]; ++i) l->bases.push_back({thread_shape[0] << i, 0});
        // thread id row-major over the thread shape (tile_i = t / cols, tile_j = t % cols)
        for (int i = 0; i < lg_t[1]; ++i) l->bases.push_back({0, 1 << i});
        for (int i = 0; i < lg_t[0]; ++i) l->bases.push_back({1 << i, 0});
        *out = l;
        return TG_OK;
    });
}

int tg_layout_swizzle128(int rows, int elem_bytes, tg_layout** out) {
    if (!out) return TG_ERR_INVALID_ARG;
    return guarded([&] {
        const int lg_rows = log2_exact(rows);
        const int lg_eb = log2_exact(elem_bytes);
        if (lg_rows < 3 || lg_eb > 3 || lg_rows > 20) throw LayoutError();
        const int lg_cols = 7 - lg_eb;  // elements per 128-byte row
        tg_layout* l = make({"offset"}, {lg_rows + lg_cols}, {"row", "col"}, {lg_rows, lg_cols});
        for (int b = 0; b < lg_rows + lg_cols; ++b) {
            const int64_t byte = (int64_t)elem_bytes << b;
            const int64_t row = byte >> 7;
            const int64_t chunk = ((byte >> 4) & 7) ^ (row & 7);
            const int64_t col = ((chunk << 4) | (byte & 15)) >> lg_eb;
            l->bases.push_back({(int32_t)row, (int32_t)col});
        }
        *out = l;
        return TG_OK;
    });
}

int tg_layout_tmem_32x32b(int bn, tg_layout** out) {
    if (!out) return TG_ERR_INVALID_ARG;
    return guarded([&] {
        const int lg_bn = log2_exact(bn);
        if (bn < 32 || bn > 256) throw LayoutError();
        tg_layout* l = make({"register", "lane", "warp"}, {lg_bn, 5, 2}, {"m", "n"}, {7, lg_bn});
        for (int i = 0; i < lg_bn; ++i) l->bases.push_back({0, 1 << i});
        for (int i = 0; i < 5; ++i) l->bases.push_back({1 << i, 0});
        for (int i = 0; i < 2; ++i) l->bases.push_back({32 << i, 0});
        *out = l;
        return TG_OK;
    });
}

int tg_layout_fold(const tg_layout* l, int n_fixed, const char* const* fixed_names,
                   const int32_t* fixed_values, tg_folded_layout* out) {
    if (!l || !out || n_fixed < 0 || (n_fixed > 0 && (!fixed_names || !fixed_values)))
        return TG_ERR_INVALID_ARG;
    return guarded([&] {
        const size_t nin = l->in_names.size(), nout = l->out_names.size();
        std::vector<int32_t> fixed(nin, 0);  // variable inputs stay 0: no part in the constant
        std::vector<char> is_fixed(nin, 0);
        for (int k = 0; k < n_fixed; ++k) {
            if (!fixed_names[k]) throw LayoutError();
            const int d = find(l->in_names, fixed_names[k]);
            if (d < 0 || is_fixed[d]) throw LayoutError();
            if (fixed_values[k] < 0 || fixed_values[k] >= (1 << l->in_bits[d])) throw LayoutError();
            is_fixed[d] = 1;
            fixed[d] = fixed_values[k];
        }
        if (nout > TG_FOLD_MAX_OUTS || total(l->out_bits) > 32) throw LayoutError();
        tg_folded_layout f;
        std::memset(&f, 0, sizeof(f));
        f.n_outs = (int)nout;
        int shift = 0;
        for (size_t o = 0; o < nout; ++o) {
            f.out_shift[o] = shift;
            f.out_bits[o] = l->out_bits[o];
            shift += l->out_bits[o];
        }
        // every output coordinate as a bit field of one word: XOR of words is
        // XOR of every coordinate at once
        auto pack = [&](const std::vector<int32_t>& c) {
            uint32_t w = 0;
            for (size_t o = 0; o < nout; ++o)
                if (f.out_bits[o] > 0) w |= (uint32_t)c[o] << f.out_shift[o];
            return w;
        };
        f.constant = pack(apply(*l, fixed.data()));
        int row = 0;
        for (size_t d = 0; d < nin; ++d) {
            if (!is_fixed[d]) {
                if (f.n_vars >= TG_FOLD_MAX_VARS || f.n_bits + l->in_bits[d] > TG_FOLD_MAX_BITS)
                    throw LayoutError();
                f.var_bits[f.n_vars++] = l->in_bits[d];
                for (int i = 0; i < l->in_bits[d]; ++i) f.cols[f.n_bits++] = pack(l->bases[row + i]);
            }
            row += l->in_bits[d];
        }
        *out = f;
        return TG_OK;
    });
}

int tg_layout_folded_apply(const tg_folded_layout* f, const int32_t* vars, int32_t* outs) {
    if (!f || (!vars && f->n_vars > 0) || (!outs && f->n_outs > 0)) return TG_ERR_INVALID_ARG;
    if (f->n_vars < 0 || f->n_vars > TG_FOLD_MAX_VARS || f->n_outs < 0 ||
        f->n_outs > TG_FOLD_MAX_OUTS || f->n_bits < 0 || f->n_bits > TG_FOLD_MAX_BITS)
        return TG_ERR_LAYOUT;
    uint32_t v[TG_FOLD_MAX_VARS] = {};
    for (int k = 0; k < f->n_vars; ++k) {
        if (f->var_bits[k] < 0 || f->var_bits[k] > 30 || vars[k] < 0 ||
            vars[k] >= (1 << f->var_bits[k]))
            return TG_ERR_INVALID_ARG;
        v[k] = (uint32_t)vars[k];
    }
    const uint32_t packed = tg_folded_apply_packed(f, v);
    for (int o = 0; o < f->n_outs; ++o) outs[o] = tg_folded_output(f, packed, o);
    return TG_OK;
}

}  // extern "C"
