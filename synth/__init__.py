"""Seeded synthetic inputs for the Kamera reuse operator (shared by the tests,
the benchmark and the oracle checks; holds none of the operator's arithmetic).

``gen``        counter-based generator (host, numpy)
``workloads``  the workload shapes (tiny MHA, GQA video, MLA, sliding window,
               long-video reorder + recall) and their host/device fills
``device``     ctypes loader of the CUDA twin of ``gen`` (synth_cuda.cu)
"""
