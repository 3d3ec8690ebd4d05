"""The ncu launch-list summariser on a small hand-written CSV."""
import json

from iteration_level_selective_gb300 import ncu_summary as ns

CSV = '''==PROF== Connected to process 1
"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"
"0","1","python","h","void orca::(anonymous namespace)::gemm_tc_bf16_kernel<128>(CUtensorMap, int)","1","7","(192, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","Mbyte","2.50"
"0","1","python","h","void orca::(anonymous namespace)::gemm_tc_bf16_kernel<128>(CUtensorMap, int)","1","7","(192, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","Kbyte","500"
"0","1","python","h","void orca::(anonymous namespace)::gemm_tc_bf16_kernel<128>(CUtensorMap, int)","1","7","(192, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","gpu__time_duration.sum","usecond","10.00"
"1","1","python","h","void orca::attention_kernel<__nv_bfloat16, 64>(orca::AttnArgs)","1","7","(256, 1, 1)","(304, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","byte","1,000,000"
"1","1","python","h","void orca::attention_kernel<__nv_bfloat16, 64>(orca::AttnArgs)","1","7","(256, 1, 1)","(304, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","byte","0"
"1","1","python","h","void orca::attention_kernel<__nv_bfloat16, 64>(orca::AttnArgs)","1","7","(256, 1, 1)","(304, 1, 1)","0","10.3","Command line profiler metrics","gpu__time_duration.sum","nsecond","30000"
"2","1","python","h","void orca::prefill_attention_tc_kernel<64>(CUtensorMap, CUtensorMap, orca::TcAttnArgs)","1","7","(128, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","byte","500000"
"2","1","python","h","void orca::prefill_attention_tc_kernel<64>(CUtensorMap, CUtensorMap, orca::TcAttnArgs)","1","7","(128, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","byte","0"
"2","1","python","h","void orca::prefill_attention_tc_kernel<64>(CUtensorMap, CUtensorMap, orca::TcAttnArgs)","1","7","(128, 1, 1)","(152, 1, 1)","0","10.3","Command line profiler metrics","gpu__time_duration.sum","usecond","60"
'''


def test_summary_and_traffic(tmp_path):
    p = tmp_path / "l.csv"
    p.write_text(CSV)
    per = ns.summarise(ns.read_launches(str(p)))
    assert set(per) == {"gemm_tc_bf16_kernel", "attention_kernel", "prefill_attention_tc_kernel"}
    g = per["gemm_tc_bf16_kernel"]
    assert g["launches"] == 1 and abs(g["ms"] - 0.010) < 1e-12 and abs(g["dram"] - 3.0e6) < 1e-6
    assert abs(per["attention_kernel"]["ms"] - 0.030) < 1e-12
    md = ns.markdown(per)
    assert "| prefill_attention_tc_kernel | 1 | 0.060 | 0.600 |" in md
    t = ns.traffic_by_class(per, scale=2.0)
    assert abs(t["gemm_tc_bf16"] - 6.0e6) < 1e-6
    assert abs(t["attention"] - 3.0e6) < 1e-6       # both attention kernels over one ragged-kernel launch
    out = tmp_path / "traffic.json"
    ns.main([str(p), "--traffic", str(out), "--workload", "w"])
    d = json.loads(out.read_text())
    assert d["w"]["gemm_tc_bf16"]["source_hash"] == ns.source_hash()


def test_gemm_class_sums_alternative_kernels(tmp_path):
    """The GEMM class divides the bytes of the persistent and the cluster
    split-K kernels by the launches of both (each Linear is one or the other)."""
    extra = '''"3","1","python","h","void orca::(anonymous namespace)::gemm_tc_cluster_kernel<64>(CUtensorMap, int)","1","7","(192, 1, 1)","(96, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","Mbyte","1.00"
"3","1","python","h","void orca::(anonymous namespace)::gemm_tc_cluster_kernel<64>(CUtensorMap, int)","1","7","(192, 1, 1)","(96, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","byte","0"
"3","1","python","h","void orca::(anonymous namespace)::gemm_tc_cluster_kernel<64>(CUtensorMap, int)","1","7","(192, 1, 1)","(96, 1, 1)","0","10.3","Command line profiler metrics","gpu__time_duration.sum","usecond","5"
'''
    p = tmp_path / "l.csv"
    p.write_text(CSV + extra)
    per = ns.summarise(ns.read_launches(str(p)))
    t = ns.traffic_by_class(per)
    assert abs(t["gemm_tc_bf16"] - (3.0e6 + 1.0e6) / 2) < 1e-6


def test_source_hash_ignores_comments_and_layout(tmp_path):
    a = tmp_path / "a"
    b = tmp_path / "b"
    a.mkdir()
    b.mkdir()
    (a / "k.cu").write_text('// header\n__global__ void k() { asm("mov.u32 %0, 1; // in a string"); }\n')
    (b / "k.cu").write_text('/* another header */\n__global__ void k()\n{\n  asm("mov.u32 %0, 1; // in a string");  // note\n}\n')
    assert ns.source_hash(str(a)) == ns.source_hash(str(b))
    (b / "k.cu").write_text('__global__ void k() { asm("mov.u32 %0, 2; // in a string"); }\n')
    assert ns.source_hash(str(a)) != ns.source_hash(str(b))
    assert ns.code_only('x = "/*"; /* c */ y = \'"\'; // d\nz') == 'x = "/*"; y = \'"\'; z'


def test_short_name_of_the_names_ncu_prints():
    assert ns.short_name("void orca::(anonymous namespace)::gemm_tc_bf16_kernel<128>(CUtensorMap, int)") == \
        "gemm_tc_bf16_kernel"
    assert ns.short_name("void orca::<unnamed>::gemm_tc_bf16_kernel<256, 1>(CUtensorMap_st, int)") == \
        "gemm_tc_bf16_kernel"
    assert ns.short_name("orca::<unnamed>::ln_fold_vectors_kernel(const __nv_bfloat16 *, int)") == \
        "ln_fold_vectors_kernel"
    assert ns.short_name("void orca::<unnamed>::gemm_tc_pair_kernel(CUtensorMap_st, CUtensorMap_st, int)") == \
        "gemm_tc_pair_kernel"
    assert ns.short_name("void orca::<unnamed>::gemm_tc_pair_kernel<true>(CUtensorMap_st, CUtensorMap_st, int)") == \
        "gemm_tc_pair_kernel"


RAW = """"ID","Kernel Name","gpu__time_duration.sum","sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed","dram__bytes_read.sum","launch__grid_size","smsp__pcsamp_warps_issue_stalled_wait","smsp__pcsamp_warps_issue_stalled_long_scoreboard","smsp__pcsamp_warps_issue_stalled_long_scoreboard_not_issued","smsp__pcsamp_warps_issue_stalled_barrier"
"","","msecond","%","Mbyte","","warp","warp","warp","warp"
"0","void orca::<unnamed>::prefill_attention_tc_kernel<128>(CUtensorMap_st, TcAttnArgs)","0.6276","31.37","788.8","152","6,699","15,273","14,000","735"
"""


def test_raw_page_summary():
    """The raw-page summary converts the units the capture states and ranks
    the sampled stall reasons (the *_not_issued subsets left out)."""
    from iteration_level_selective_gb300 import ncu_summary as ns
    t = ns.raw_summary(RAW)
    lines = t.splitlines()
    assert lines[0] == "| metric | prefill_attention_tc_kernel |"
    row = {l.split("|")[1].strip(): l.split("|")[2].strip() for l in lines[2:]}
    assert row["duration (us)"] == "627.6"
    assert row["DRAM read (GB)"] == "0.7888"
    assert row["tensor pipe active, % of elapsed"] == "31.37 %"
    assert row["grid"] == "152"
    assert row["top sampled stall reasons"] == "long_scoreboard 15273, wait 6699, barrier 735"
