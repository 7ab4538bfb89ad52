"""The benchmark's roofline byte accounting against the oracle: the algorithmic bytes
one decode-attention launch moves must equal the size of the packed state the oracle
builds for the same tokens (codes, metadata, the valid residual rows), plus the queries
read and the outputs written. CPU only."""

import dataclasses

import pytest

import bench
import oracle
import synth

NAMES = ["llama8b-int8", "kivi-int4", "kivi-int2", "kivi-k8v4", "long-int4-16k", "sym8-b16", "sym8o4-b16",
         "kivi-int4o4"]


@pytest.mark.parametrize("name", NAMES)
@pytest.mark.parametrize("T", [2 * 137, 512, 2 * 300])
def test_attention_bytes_equal_the_oracle_state(name, T):
    w = dataclasses.replace(synth.WORKLOADS[name], batch=1, n_kv=1, seq=T, steps=0)
    d = w.d_head
    k = synth.k_slice(w, 0, 0, 0, range(T))
    v = synth.v_slice(w, 0, 0, 0, range(T))
    if w.symmetric:
        st = oracle.cache_state_sym(k, v, d=d, k_outliers=w.k_outliers)
    else:
        st = oracle.cache_state(k, v, d=d, bits=w.bits, G=w.k_group, Gv=w.v_group, R=w.residual, v_bits=w.vbits,
                                k_outliers=w.k_outliers)
    state = (st.k_codes.nbytes + st.k_meta.nbytes + (T - st.Tq) * d * 2 + st.v_codes.nbytes
             + st.v_meta.nbytes + (st.k_sparse.nbytes if st.k_sparse is not None else 0))
    io = w.n_q * d * 2 + w.n_q * d * 4  # binary16 queries in, binary32 outputs out
    assert bench.attn_bytes_per_layer(w, T) == state + io


@pytest.mark.parametrize("name", NAMES)
def test_prefill_bytes_equal_inputs_plus_state(name):
    T = 2 * 300
    w = dataclasses.replace(synth.WORKLOADS[name], batch=1, n_kv=1, seq=T, steps=0)
    d = w.d_head
    k = synth.k_slice(w, 0, 0, 0, range(T))
    v = synth.v_slice(w, 0, 0, 0, range(T))
    if w.symmetric:
        st = oracle.cache_state_sym(k, v, d=d, k_outliers=w.k_outliers)
    else:
        st = oracle.cache_state(k, v, d=d, bits=w.bits, G=w.k_group, Gv=w.v_group, R=w.residual, v_bits=w.vbits,
                                k_outliers=w.k_outliers)
    written = (st.k_codes.nbytes + st.k_meta.nbytes + (T - st.Tq) * d * 2 + st.v_codes.nbytes
               + st.v_meta.nbytes + (st.k_sparse.nbytes if st.k_sparse is not None else 0))
    assert bench.prefill_bytes_per_layer(w, T) == 2 * T * d * 2 + written
