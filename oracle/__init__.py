"""fp64 CPU oracle for the MiniMax Sparse Attention (MSA) decode path.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
baseline use this package; the library's own code path never imports it, and it
imports nothing from the library (it shares no kernels, helpers or constants
with the CUDA code). It is written to be read against the pages, not to be fast:
plain numpy in fp64, following the method's steps in the order the pages give
them.

Sources (page title, section):
  * "MiniMax-M3.1-Flash Day-0 対応" (aisoku.org; the extraction has no title
    line, so the page is named by its subject), section "MSAの仕組み":
    128-token KV blocks, a light indexer picks the top blocks plus the most
    recent block, exact attention over those blocks only, at most 2,048 keys per
    query; section "何が新しいか": NVFP4 KV at 34,560 bytes/token vs 61,440 for
    FP8.
  * "MiniMax M3 vLLM サポート：1M トークンマルチモーダル推論の Day-0 サービング"
    (agentlenshq.com), section "MSA 実行プロセス":
    1) block scoring by a small index head, 2) top-k block selection with
    local_blocks=1, 3) sparse GQA with online softmax; section "EAGLE3 を用いた
    投機的デコード": a decode-only split-K path with a unified decode_query_len.
  * "vLLM、AMD Instinct MI355X上でMiniMax M3のボトルネック最適化手法を公開"
    (news.ainew.jp), question 1: 64 query heads,
    4 KV heads, 4 index heads; question 2: the indexer handles all draft
    positions of a request together and drops the positive score scale, since a
    positive constant does not change the top-k order.

Modules: ``formats`` (bf16 / E4M3 / E2M1 / NVFP4 from their definitions),
``quant`` (cache insertion and quantisation), ``msa`` (scores, selection,
sparse and dense attention).

Parity status: every function here is pinned by tests/test_oracle_*.py against
hand-worked examples, closed forms, library routines or invariants.
"""
